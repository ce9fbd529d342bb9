"""Prefix-cache state checkpoints (kda_chunk_fwd_checkpoints) vs the oracle (needs a GPU).

K3 explainer, section 14 "Prefix Cache": a cached prefix is resumed from the KDA
state saved at a reusable boundary. Slot (s, i) must equal the state of sequence s
after its first (i + 1) * every tokens: the oracle's state with t_stop at that
boundary, and bitwise the final state of a kda_chunk_fwd call over just the prefix.
Slots whose boundary lies past a sequence's end are left untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from util import TOL, np32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = 1234.5
TOKEN_KEYS = ("q", "k", "v", "log_alpha", "beta", "gate")


def _oracle_states_at(x, cu, stops, S0, scale):
    g = None if x["gate"] is None else np32(x["gate"])
    s0 = None if S0 is None else np32(S0).astype(np.float64)
    _, st = oracle.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                           np32(x["beta"]), g, s0, list(cu), scale=scale, t_stop=stops)
    return st


def _run_ckpt(x, cu_t, n_seq, S0, every, per, scale=1.0):
    T, H, dk = x["k"].shape
    dv = x["v"].shape[-1]
    out = torch.empty((T, H, dv), dtype=x["v"].dtype, device=DEV)
    fs = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=DEV)
    ck = torch.full((n_seq, per, H, dk, dv), SENTINEL, dtype=torch.float32, device=DEV)
    B.kda_chunk_fwd_checkpoints(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                                out, S0, fs, ck, every, cu_t, n_seq, scale=scale)
    assert B.kda_get_error() == B.KDA_OK
    return out, fs, ck


@pytest.mark.parametrize("dk,dv,dtype", [
    (128, 128, torch.bfloat16),  # tensor-core path
    (128, 128, torch.float32),
    (64, 64, torch.bfloat16),
    (64, 128, torch.float32),
])
def test_checkpoints_ragged_vs_oracle(dk, dv, dtype):
    """Lengths around every boundary case (empty, shorter than one spacing, exactly
    one, a ragged tail, more boundaries than slots); spacing 128 tokens, 6 slots."""
    lengths = [0, 1, 127, 128, 200, 384, 700, 1029]
    every, per, H, scale = 128, 6, 2, 0.7
    T = sum(lengths)
    cu = [0] + np.cumsum(lengths).tolist()
    n_seq = len(lengths)
    x = inputs.tokens(T, H, dk, dv, dtype, seed=31, device=DEV)
    S0 = inputs.state(n_seq, H, dk, dv, seed=32, device=DEV)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out, fs, ck = _run_ckpt(x, cu_t, n_seq, S0, every, per, scale)
    # the checkpoint output changes nothing else, bit for bit
    out0, fs0 = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0,
                            cu_t, n_seq=n_seq, scale=scale)
    assert torch.equal(out, out0) and torch.equal(fs, fs0)
    tol = TOL[dtype]
    ck_h = ck.cpu().numpy()
    for i in range(per):
        b = (i + 1) * every
        ref = _oracle_states_at(x, cu, [min(b, L) for L in lengths], S0, scale)
        for s, L in enumerate(lengths):
            if b <= L:
                e = rel_err(ck_h[s, i], ref[s])
                assert e <= tol, (s, i, e)
            else:
                assert np.all(ck_h[s, i] == SENTINEL), (s, i)
    # a boundary at a sequence's end is its final state
    s128 = lengths.index(128)
    assert torch.equal(ck[s128, 0], fs[s128])


def test_checkpoints_prefill_workload_bitwise_prefix():
    """4 x 4096 tokens, 16 heads, d = 128, bf16, S0 ~ N(0, 0.01), a checkpoint every
    1024 tokens: each checkpoint is bitwise the final state of the same sequences cut
    after that many tokens, and the first one matches the oracle."""
    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device=DEV)
    n_seq, L, every = len(w.lengths), w.lengths[0], 1024
    per = L // every
    out, fs, ck = _run_ckpt(x, None, n_seq, x["S0"], every, per)
    assert torch.equal(ck[:, per - 1], fs)
    for i in range(per - 1):
        P = (i + 1) * every
        # the first P tokens of every sequence, packed (token tensors only)
        xp = {k: torch.cat([x[k][s * L:s * L + P] for s in range(n_seq)]).contiguous()
              for k in TOKEN_KEYS}
        _, fsp = B.chunk_fwd(xp["q"], xp["k"], xp["v"], xp["log_alpha"], xp["beta"],
                             xp["gate"], x["S0"], None, n_seq=n_seq)
        assert torch.equal(ck[:, i], fsp), i
    ref = _oracle_states_at(x, w.cu_seqlens, [every] * n_seq, x["S0"], 1.0)
    assert rel_err(np32(ck[:, 0]), ref) <= TOL[torch.bfloat16]
