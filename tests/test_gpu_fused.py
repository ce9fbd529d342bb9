"""The persistent prefill (one cooperative launch) against the two-kernel schedule and the
oracle (needs a GPU).

Fixed-length batches with few (sequence, head) chains (at most 48, each of at least 16 chunks)
run cards and state pass in one launch:
every CTA first builds update cards in chunk-major order, then the chain owners walk their
chains while the others keep building (K3 training analysis, section 4: FlashKDA overlaps the
intra-chunk computation with the cross-chunk state propagation). Each card and each chain is
computed by the same code as in the two-kernel schedule, so the results must match that
schedule (reached by passing the same lengths as cu_seqlens) bit for bit, and the oracle
within the bf16 tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from util import TOL, check, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


def _run(x, S0, n_seq, cu=None, final=True, flags=B.KDA_QK_L2NORM, scale=1.0):
    T, H, _ = x["v"].shape
    out = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    fs = torch.full((n_seq, H, D, D), float("nan"), device=DEV) if final else None
    B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, S0, fs,
                    cu, n_seq, scale=scale, flags=flags)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    return out, fs


@pytest.mark.parametrize("n_seq,L,H", [
    (1, 1024, 1),    # a single chain of 16 chunks
    (3, 1333, 5),    # ragged last chunk (53 tokens), 15 chains
    (2, 4096, 16),   # 32 chains of 64 chunks
    (3, 1024, 16),   # 48 chains: the most the persistent prefill takes
])
def test_fused_equals_two_kernel_schedule_and_oracle(n_seq, L, H):
    T = n_seq * L
    assert B.kda_chunk_fwd_launches(T, n_seq, H, D, D) == 1
    x = inputs.tokens(T, H, D, D, torch.bfloat16, seed=700 + L, device=DEV)
    S0 = inputs.state(n_seq, H, D, D, seed=701 + L, device=DEV)
    o_f, s_f = _run(x, S0, n_seq, scale=0.7)
    cu = torch.arange(0, T + 1, L, dtype=torch.int32, device=DEV)
    o_v, s_v = _run(x, S0, n_seq, cu=cu, scale=0.7)
    assert torch.equal(o_f, o_v)
    assert torch.equal(s_f, s_v)
    for s, h in ((0, 0), (n_seq - 1, H - 1)):
        rows = slice(s * L, (s + 1) * L)
        g = lambda t: np32(t[rows, h:h + 1])
        ro, rs = oracle.forward(g(x["q"]), g(x["k"]), g(x["v"]), g(x["log_alpha"]),
                                np32(x["beta"][rows, h:h + 1]), g(x["gate"]),
                                np32(S0[s:s + 1, h:h + 1]).astype(np.float64), [0, L], scale=0.7)
        check(f"fused/{n_seq}x{L}x{H}/out_seq{s}_head{h}", np32(o_f[rows, h:h + 1]), ro,
              TOL[torch.bfloat16])
        check(f"fused/{n_seq}x{L}x{H}/state_seq{s}_head{h}", np32(s_f[s:s + 1, h:h + 1]), rs,
              TOL[torch.bfloat16])


def test_fused_without_state_buffers_and_with_gate_logits():
    """No initial or final state, gate and beta as logits: still bitwise the two-kernel call."""
    n_seq, L, H = 2, 1100, 8
    T = n_seq * L
    x = inputs.tokens(T, H, D, D, torch.bfloat16, seed=720, device=DEV)
    flags = B.KDA_QK_L2NORM | B.KDA_GATE_LOGITS
    o_f, _ = _run(x, None, n_seq, final=False, flags=flags)
    cu = torch.arange(0, T + 1, L, dtype=torch.int32, device=DEV)
    o_v, _ = _run(x, None, n_seq, cu=cu, final=False, flags=flags)
    assert torch.equal(o_f, o_v)
    assert torch.isfinite(o_f.float()).all()


def test_fused_repeated_calls_are_bitwise_equal():
    """The flags and the card counter are reset by every call: a second call on the same
    workspace gives the same bits."""
    n_seq, L, H = 2, 8192, 16
    T = n_seq * L
    x = inputs.tokens(T, H, D, D, torch.bfloat16, seed=730, device=DEV)
    S0 = inputs.state(n_seq, H, D, D, seed=731, device=DEV)
    ws = torch.empty(B.kda_chunk_fwd_workspace_size(T, n_seq, H, D, D), dtype=torch.uint8,
                     device=DEV)
    res = []
    for _ in range(3):
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
        fs = torch.empty((n_seq, H, D, D), device=DEV)
        B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, S0,
                        fs, None, n_seq, workspace=ws)
        res.append((out, fs))
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    for out, fs in res[1:]:
        assert torch.equal(out, res[0][0]) and torch.equal(fs, res[0][1])
