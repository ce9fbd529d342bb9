"""Seeded random shapes through every forward schedule and the backward, against the oracles
(needs a GPU).

Each case draws its own lengths, heads, head dims, dtype, gate / L2-norm / initial-state
options and scale from a fixed seed, so a failure names a reproducible case. The cases rotate
over four kinds so that every schedule is reached: fixed lengths of 16+ chunks (the persistent
prefill or the split schedule), packed sequences of 16+ chunks (the split schedule), packed
mixes of short and ragged sequences, and short fixed lengths. Metric and tolerances as in the
other parity tests: max|gpu - ref| / max|ref| per output, fp32 <= 1e-4, bf16 <= 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from oracle import autograd as AG
from util import TOL, np32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
SHAPES = [(64, 64), (128, 128), (64, 128), (128, 64)]


def _draw(i):
    """Case i: (lengths, fixed, H, dk, dv, dtype, scale, gate, l2norm, with_init)."""
    rng = np.random.default_rng(9000 + i)
    kind = i % 4
    dk, dv = SHAPES[1] if rng.random() < 0.5 else SHAPES[int(rng.integers(0, 4))]
    tc = (dk, dv) == (128, 128)
    dtype = torch.bfloat16 if (tc and rng.random() < 0.75) or rng.random() < 0.3 else torch.float32
    if kind == 0:  # fixed lengths, 16+ chunks
        n_seq, H = int(rng.integers(1, 5)), int(rng.integers(1, 9))
        L = int(64 * rng.integers(16, 40) + rng.integers(-1, 2))
        lengths, fixed = [L] * n_seq, True
    elif kind == 1:  # packed, 16+ chunks on average
        n_seq, H = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        lengths = [int(rng.integers(1000, 3200)) for _ in range(n_seq)]
        if n_seq > 1:  # one short or empty sequence among them
            lengths[int(rng.integers(0, n_seq))] = int(rng.choice([0, 1, 65]))
        fixed = False
    elif kind == 2:  # packed mix of short and ragged sequences
        n_seq, H = int(rng.integers(2, 9)), int(rng.integers(1, 7))
        lengths = [int(rng.choice([0, 1, 63, 64, 65, 127, 129, int(rng.integers(1, 700))]))
                   for _ in range(n_seq)]
        fixed = False
    else:  # short fixed lengths
        n_seq, H = int(rng.integers(1, 7)), int(rng.integers(1, 7))
        L = int(rng.integers(1, 500))
        lengths, fixed = [L] * n_seq, True
    scale = float(rng.choice([1.0, 0.8, 0.125]))
    gate, l2norm, with_init = rng.random() < 0.8, rng.random() < 0.8, rng.random() < 0.7
    return lengths, fixed, H, dk, dv, dtype, scale, gate, l2norm, with_init


def _case_id(i):
    lengths, fixed, H, dk, dv, dtype, *_ = _draw(i)
    kind = "fixed" if fixed else "packed"
    return f"{i}-{kind}{len(lengths)}x{max(lengths)}-H{H}-{dk}x{dv}-{str(dtype)[6:]}"


def _inputs(i):
    lengths, fixed, H, dk, dv, dtype, scale, gate, l2norm, with_init = _draw(i)
    T = sum(lengths)
    x = inputs.tokens(T, H, dk, dv, dtype, seed=9100 + i, device=DEV)
    if not gate:
        x["gate"] = None
    S0 = inputs.state(len(lengths), H, dk, dv, seed=9200 + i, device=DEV) if with_init else None
    cu = [0] + np.cumsum(lengths).tolist()
    return x, S0, cu, fixed, dtype, scale, l2norm


@pytest.mark.parametrize("i", range(48), ids=_case_id)
def test_forward_random_case(i):
    x, S0, cu, fixed, dtype, scale, l2norm = _inputs(i)
    n_seq = len(cu) - 1
    cu_t = None if fixed else torch.tensor(cu, dtype=torch.int32, device=DEV)
    out, fs = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0, cu_t,
                          n_seq=n_seq, scale=scale, l2norm=l2norm)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    g = None if x["gate"] is None else np32(x["gate"])
    s0 = None if S0 is None else np32(S0).astype(np.float64)
    ro, rs = oracle.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                            np32(x["beta"]), g, s0, cu, scale=scale, l2norm=l2norm)
    if out.numel():
        assert rel_err(np32(out), ro) <= TOL[dtype]
    assert rel_err(np32(fs), rs) <= TOL[dtype]


@pytest.mark.parametrize("i", [2, 6, 9, 10, 14, 18, 22, 27], ids=_case_id)
def test_backward_random_case(i):
    x, S0, cu, fixed, dtype, scale, l2norm = _inputs(i)
    n_seq = len(cu) - 1
    T, H, dv = x["v"].shape
    dk = x["k"].shape[-1]
    gen = torch.Generator(device="cpu").manual_seed(9300 + i)
    d_out = torch.randn((T, H, dv), generator=gen).to(dtype).to(DEV)
    d_fin = torch.randn((n_seq, H, dk, dv), generator=gen).to(DEV)
    cu_t = None if fixed else torch.tensor(cu, dtype=torch.int32, device=DEV)
    got = B.chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0, d_out,
                      d_fin, cu_t, n_seq=n_seq, scale=scale, l2norm=l2norm)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    f = lambda t: None if t is None else np32(t)
    ref = AG.backward(f(x["q"]), f(x["k"]), f(x["v"]), f(x["log_alpha"]), f(x["beta"]),
                      f(x["gate"]), f(S0), cu, f(d_out), f(d_fin), scale=scale, l2norm=l2norm)
    for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dgate", "dS0"):
        if ref.get(n) is None:
            assert got.get(n) is None, n
            continue
        if got[n].numel():
            assert rel_err(np32(got[n]), ref[n]) <= TOL[dtype], n
