"""Split prefill (tensor-core path) against the oracle and the unsplit schedule (needs a GPU).

With few (sequence, head) pairs and long sequences, kda_chunk_fwd builds the cards of each
sequence's leading 12/16 of chunks, runs the state pass over them while
the cards of the trailing chunks are built, and finishes with a state pass over the trailing
chunks. The chunked algebra is unchanged (K3 training overview, section 4 "FlashKDA": the
cards are independent per chunk, only the state hand-off is ordered), so the results must
equal the oracle within the bf16 tolerance and the unsplit schedule bit for bit. The
unsplit schedule is reached without a switch: appending empty sequences lowers the average
sequence length below the split threshold and leaves every other sequence's result alone.
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
H, D = 2, 128
# empty, 1 token, one chunk + 1, ragged tails, 33+ chunks: 8280 tokens in 7 sequences
LENGTHS = [0, 1, 65, 1100, 2113, 3001, 2000]


def _problem(lengths, seed):
    T = sum(lengths)
    cu = [0] + np.cumsum(lengths).tolist()
    x = inputs.tokens(T, H, D, D, torch.bfloat16, seed=seed, device=DEV)
    S0 = inputs.state(len(lengths), H, D, D, seed=seed + 1, device=DEV)
    return x, S0, cu


def _run(x, S0, cu, every=None, per=0, scale=0.8):
    T = x["k"].shape[0]
    n_seq = len(cu) - 1
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    fs = torch.empty((n_seq, H, D, D), dtype=torch.float32, device=DEV)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    ck = None
    if per:
        ck = torch.full((n_seq, per, H, D, D), -7.0, dtype=torch.float32, device=DEV)
        B.kda_chunk_fwd_checkpoints(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                    x["gate"], out, S0, fs, ck, every, cu_t, n_seq, scale=scale)
    else:
        B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, S0,
                        fs, cu_t, n_seq, scale=scale)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    return out, fs, ck


def _padded(S0, cu, extra):
    """The same problem with `extra` empty sequences appended."""
    S0p = torch.cat([S0, torch.zeros((extra, H, D, D), dtype=S0.dtype, device=DEV)])
    return S0p, cu + [cu[-1]] * extra


def test_schedules_are_as_intended():
    T, n = sum(LENGTHS), len(LENGTHS)
    assert B.kda_chunk_fwd_launches(T, n, H, D, D, varlen=True) == 5
    assert B.kda_chunk_fwd_launches(T, n + 2, H, D, D, varlen=True) == 3


def test_split_vs_oracle():
    x, S0, cu = _problem(LENGTHS, 61)
    out, fs, _ = _run(x, S0, cu)
    ro, rs = oracle.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                            np32(x["beta"]), np32(x["gate"]), np32(S0).astype(np.float64), cu,
                            scale=0.8)
    assert rel_err(np32(out), ro) <= TOL[torch.bfloat16]
    assert rel_err(np32(fs), rs) <= TOL[torch.bfloat16]


def test_split_bitwise_equals_unsplit():
    x, S0, cu = _problem(LENGTHS, 62)
    out_s, fs_s, _ = _run(x, S0, cu)
    S0p, cup = _padded(S0, cu, 2)
    out_u, fs_u, _ = _run(x, S0p, cup)
    assert torch.equal(out_s, out_u)
    assert torch.equal(fs_s, fs_u[:len(LENGTHS)])
    # the appended empty sequences hand their zero entry state straight through
    assert torch.count_nonzero(fs_u[len(LENGTHS):]) == 0


def test_split_checkpoints_bitwise_equal_unsplit():
    """Checkpoints every 512 tokens (slots on both sides of every split point)."""
    x, S0, cu = _problem(LENGTHS, 63)
    out_s, fs_s, ck_s = _run(x, S0, cu, every=512, per=6)
    S0p, cup = _padded(S0, cu, 2)
    out_u, fs_u, ck_u = _run(x, S0p, cup, every=512, per=6)
    n = len(LENGTHS)
    assert torch.equal(out_s, out_u)
    assert torch.equal(fs_s, fs_u[:n])
    assert torch.equal(ck_s, ck_u[:n])
    # a slot is written exactly when its boundary lies inside the sequence
    for s, L in enumerate(LENGTHS):
        for i in range(6):
            written = not torch.all(ck_s[s, i] == -7.0)
            assert written == ((i + 1) * 512 <= L), (s, i)


def test_split_prefill_workload_bitwise_and_sampled():
    """The bench workload (4 x 4096 tokens, 16 heads) takes the split; it equals the same
    sequences run unsplit, and the oracle on two sampled (sequence, head) chains."""
    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device=DEV)
    n_seq, L, Hw = len(w.lengths), w.lengths[0], w.H
    T = n_seq * L
    assert B.kda_chunk_fwd_launches(T, n_seq, Hw, D, D) == 4  # fixed lengths: no chunk table
    out = torch.empty((T, Hw, D), dtype=torch.bfloat16, device=DEV)
    fs = torch.empty((n_seq, Hw, D, D), dtype=torch.float32, device=DEV)
    B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, x["S0"],
                    fs, None, n_seq)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    # unsplit: the same four sequences plus four empty ones (8 x 16 pairs > 112)
    cu = [s * L for s in range(n_seq + 1)] + [T] * 4
    assert B.kda_chunk_fwd_launches(T, n_seq + 4, Hw, D, D, varlen=True) == 3
    out_u = torch.empty_like(out)
    fs_u = torch.empty((n_seq + 4, Hw, D, D), dtype=torch.float32, device=DEV)
    S0p = torch.cat([x["S0"], torch.zeros((4, Hw, D, D), dtype=torch.float32, device=DEV)])
    B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out_u, S0p,
                    fs_u, torch.tensor(cu, dtype=torch.int32, device=DEV), n_seq + 4)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(out, out_u)
    assert torch.equal(fs, fs_u[:n_seq])
    for s, h in ((0, 3), (3, 14)):
        rows = slice(s * L, (s + 1) * L)
        g = lambda t: np32(t[rows, h:h + 1])
        ro, rs = oracle.forward(g(x["q"]), g(x["k"]), g(x["v"]), g(x["log_alpha"]),
                                np32(x["beta"][rows, h:h + 1]), g(x["gate"]),
                                np32(x["S0"][s:s + 1, h:h + 1]).astype(np.float64), [0, L])
        assert rel_err(np32(out[rows, h:h + 1]), ro) <= TOL[torch.bfloat16]
        assert rel_err(np32(fs[s:s + 1, h:h + 1]), rs) <= TOL[torch.bfloat16]


def test_fixed_length_split_checkpoints_equal_prefix_calls():
    """The bench workload (no cu_seqlens: closed-form indexing, split after chunk 48) with a
    checkpoint every 1024 tokens. Each slot equals, bit for bit, the final state of a call over
    just that prefix of every sequence (the slots after chunk 63 of the trailing part and after
    chunks 15, 31, 47 of the leading one)."""
    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device=DEV)
    n_seq, L, Hw = len(w.lengths), w.lengths[0], w.H
    T, every, per = n_seq * L, 1024, L // 1024
    out = torch.empty((T, Hw, D), dtype=torch.bfloat16, device=DEV)
    fs = torch.empty((n_seq, Hw, D, D), dtype=torch.float32, device=DEV)
    ck = torch.full((n_seq, per, Hw, D, D), -7.0, dtype=torch.float32, device=DEV)
    B.kda_chunk_fwd_checkpoints(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                                out, x["S0"], fs, ck, every, None, n_seq)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(ck[:, per - 1], fs)
    for i in range(per - 1):
        P = every * (i + 1)
        xp = {n: x[n].view(n_seq, L, *x[n].shape[1:])[:, :P].reshape(n_seq * P, *x[n].shape[1:])
              for n in ("q", "k", "v", "log_alpha", "beta", "gate")}
        fp = torch.empty_like(fs)
        op = torch.empty((n_seq * P, Hw, D), dtype=torch.bfloat16, device=DEV)
        B.kda_chunk_fwd(xp["q"], xp["k"], xp["v"], xp["log_alpha"], xp["beta"], xp["gate"], op,
                        x["S0"], fp, None, n_seq)
        torch.cuda.synchronize()
        assert B.kda_get_error() == B.KDA_OK
        assert torch.equal(ck[:, i], fp), i
        assert torch.equal(op.view(n_seq, P, Hw, D), out.view(n_seq, L, Hw, D)[:, :P]), i
