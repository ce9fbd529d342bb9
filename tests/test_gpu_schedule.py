"""Chain scheduling of the tensor-core state pass (needs a GPU).

The chunk table orders the sequences longest first (up to 256 of them; beyond that in index
order), and the state pass's CTAs take the (sequence, head) chains in that order. Every chain
is computed the same way wherever it lands, so a sequence's output and final state must not
depend on the batch it is part of, or on its place in it: bitwise. The chunked algebra is the
FlashKDA split of the K3 training overview, section 4; the oracle is the plain recurrence.
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
D = 128


def _run(x, S0, lengths, H):
    T = sum(lengths)
    cu = torch.tensor([0] + np.cumsum(lengths).tolist(), dtype=torch.int32, device=DEV)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    fs = torch.empty((len(lengths), H, D, D), dtype=torch.float32, device=DEV)
    B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, S0, fs, cu,
                    len(lengths))
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    return out, fs


def _slice(x, t0, t1):
    return {n: (None if t is None else t[t0:t1].contiguous()) for n, t in x.items()
            if n in ("q", "k", "v", "log_alpha", "beta", "gate")}


def test_result_independent_of_batch_and_position():
    """Shortest-first lengths (the table reverses them) with 80 heads, so the 320 chains
    take three waves of CTAs; each sequence run alone must give the same bits."""
    lengths, H = [65, 300, 1000, 2500], 80
    T = sum(lengths)
    x = inputs.tokens(T, H, D, D, torch.bfloat16, seed=71, device=DEV)
    S0 = inputs.state(len(lengths), H, D, D, seed=72, device=DEV)
    out, fs = _run(x, S0, lengths, H)
    t0 = 0
    for s, L in enumerate(lengths):
        o1, f1 = _run(_slice(x, t0, t0 + L), S0[s:s + 1].contiguous(), [L], H)
        assert torch.equal(out[t0:t0 + L], o1), s
        assert torch.equal(fs[s:s + 1], f1), s
        t0 += L


def test_many_sequences_index_order_vs_oracle():
    """300 sequences (beyond the ordered range) of 0-150 tokens, one head."""
    rng = np.random.default_rng(73)
    lengths = rng.integers(0, 151, size=300).tolist()
    H = 1
    T = sum(lengths)
    x = inputs.tokens(T, H, D, D, torch.bfloat16, seed=74, device=DEV)
    S0 = inputs.state(len(lengths), H, D, D, seed=75, device=DEV)
    out, fs = _run(x, S0, lengths, H)
    cu = [0] + np.cumsum(lengths).tolist()
    ro, rs = oracle.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                            np32(x["beta"]), np32(x["gate"]), np32(S0).astype(np.float64), cu)
    assert rel_err(np32(out), ro) <= TOL[torch.bfloat16]
    assert rel_err(np32(fs), rs) <= TOL[torch.bfloat16]
