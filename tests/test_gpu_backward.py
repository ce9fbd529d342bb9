"""kda_chunk_bwd against the fp64 autograd oracle (needs a GPU).

Metric: max|gpu - ref| / max|ref| per gradient tensor; fp32 inputs <= 1e-4,
bf16 inputs (fp32 arithmetic, bf16-rounded gradients) <= 2e-2.
"""
import numpy as np
import pytest
import torch

from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from oracle import autograd as AG
from util import TOL, np32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
GRADS = ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dgate", "dS0")


def _cotangents(T, n_seq, H, dk, dv, dtype, seed, final=True):
    g = torch.Generator(device="cpu").manual_seed(seed)
    d_out = torch.randn((T, H, dv), generator=g).to(dtype).to(DEV)
    d_fin = torch.randn((n_seq, H, dk, dv), generator=g).to(DEV) if final else None
    return d_out, d_fin


def _oracle(x, S0, cu, d_out, d_fin, scale, l2norm, heads=None, rows=None):
    def sel(t):
        if t is None:
            return None
        a = np32(t)
        if rows is not None:
            a = a[rows]
        return a if heads is None else a[:, heads]

    s0 = None if S0 is None else (np32(S0) if heads is None else np32(S0)[:, heads])
    dfin = None if d_fin is None else (np32(d_fin) if heads is None else np32(d_fin)[:, heads])
    return AG.backward(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["log_alpha"]),
                       sel(x["beta"]), sel(x["gate"]), s0, cu, sel(d_out), dfin, scale=scale,
                       l2norm=l2norm)


def _check(got, ref, tol, names=GRADS):
    for n in names:
        if ref.get(n) is None:
            assert got.get(n) is None, n
            continue
        e = rel_err(np32(got[n]), ref[n])
        assert e <= tol, (n, e)


@pytest.mark.parametrize("dk,dv,dtype", [
    (128, 128, torch.bfloat16),
    (128, 128, torch.float32),
    (64, 64, torch.bfloat16),
    (64, 128, torch.float32),
    (128, 64, torch.float32),
])
def test_backward_ragged_vs_autograd(dk, dv, dtype):
    """Lengths hitting every tail case (empty, 1, 63, 64, 65, 130, 200), 2 heads, random
    initial state and final-state cotangent, gate on, L2 norm on, scale 0.8."""
    lengths = [0, 1, 63, 64, 65, 130, 200]
    H, scale = 2, 0.8
    T = sum(lengths)
    cu = [0] + np.cumsum(lengths).tolist()
    x = inputs.tokens(T, H, dk, dv, dtype, seed=41, device=DEV)
    S0 = inputs.state(len(lengths), H, dk, dv, seed=42, device=DEV)
    d_out, d_fin = _cotangents(T, len(lengths), H, dk, dv, dtype, 43)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    got = B.chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0, d_out,
                      d_fin, cu_t, scale=scale)
    assert B.kda_get_error() == B.KDA_OK
    ref = _oracle(x, S0, cu, d_out, d_fin, scale, True)
    _check(got, ref, TOL[dtype])


@pytest.mark.parametrize("d", [64, 128])
def test_backward_without_gate_norm_or_states(d):
    """No gate (no dgate), no L2 norm, zero initial state, no final-state cotangent,
    fixed-length sequences (cu_seqlens NULL); d = 128 takes the tensor-core reverse pass."""
    H, dk, dv, n_seq, L = 3, d, d, 2, 160
    x = inputs.tokens(n_seq * L, H, dk, dv, torch.float32, seed=44, device=DEV, with_gate=False)
    d_out, _ = _cotangents(n_seq * L, n_seq, H, dk, dv, torch.float32, 45, final=False)
    got = B.chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, None, d_out,
                      None, None, n_seq=n_seq, scale=1.1, l2norm=False)
    assert B.kda_get_error() == B.KDA_OK
    ref = _oracle(x, None, [0, L, 2 * L], d_out, None, 1.1, False)
    _check(got, ref, TOL[torch.float32])


def test_backward_prefill_workload_truncated_cotangent():
    """4 x 4096 tokens, 16 heads, d = 128, bf16, S0 ~ N(0, 0.01), with d_out non-zero on
    the first 200 tokens of each sequence only and no final-state cotangent. Every
    gradient of a later token is exactly zero (they cannot reach the loss), and the
    earlier ones equal the oracle's gradients of the 200-token prefix problem (heads 0
    and 9)."""
    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device=DEV)
    n_seq, L, H, d, P = len(w.lengths), w.lengths[0], w.H, w.dk, 200
    d_out, _ = _cotangents(n_seq * L, n_seq, H, d, d, torch.bfloat16, 46, final=False)
    keep = torch.zeros(n_seq * L, dtype=torch.bool, device=DEV)
    for s in range(n_seq):
        keep[s * L:s * L + P] = True
    d_out[~keep] = 0
    got = B.chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"],
                      d_out, None, None, n_seq=n_seq)
    assert B.kda_get_error() == B.KDA_OK
    for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dgate"):
        assert torch.count_nonzero(got[n][~keep]) == 0, n
    heads = [0, 9]
    rows = np.concatenate([np.arange(s * L, s * L + P) for s in range(n_seq)])
    cu = [s * P for s in range(n_seq + 1)]
    ref = _oracle(x, x["S0"], cu, d_out, None, 1.0, True, heads=heads, rows=rows)
    sub = {n: (None if got[n] is None else got[n][torch.from_numpy(rows).to(DEV)][:, heads])
           for n in GRADS if n != "dS0"}
    sub["dS0"] = got["dS0"][:, heads]
    _check(sub, ref, TOL[torch.bfloat16])


def test_backward_repeatable_bitwise():
    lengths = [100, 37]
    T, H, d = sum(lengths), 2, 128
    x = inputs.tokens(T, H, d, d, torch.bfloat16, seed=47, device=DEV)
    d_out, d_fin = _cotangents(T, 2, H, d, d, torch.bfloat16, 48)
    cu_t = torch.tensor([0, 100, 137], dtype=torch.int32, device=DEV)
    a = B.chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], None, d_out,
                    d_fin, cu_t)
    b = B.chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], None, d_out,
                    d_fin, cu_t)
    for n in GRADS:
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("d,varlen", [(128, True), (128, False), (64, True)])
def test_backward_all_sequences_empty(d, varlen):
    """T_total = 0 with three sequences: every chain is empty, so the cotangent of the initial
    state is that of the final state, unchanged (a product over zero transitions), and no
    kernel touches a token row (the token tensors have none)."""
    n_seq, H = 3, 2
    dt = torch.bfloat16 if d == 128 else torch.float32
    tok = lambda w: torch.empty((0, H, w), dtype=dt, device=DEV)
    x = {"q": tok(d), "k": tok(d), "v": tok(d), "log_alpha": tok(d), "gate": tok(d),
         "beta": torch.empty((0, H), dtype=dt, device=DEV)}
    S0 = inputs.state(n_seq, H, d, d, seed=71, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(72)
    d_fin = torch.randn((n_seq, H, d, d), generator=g).to(DEV)
    cu = torch.zeros(n_seq + 1, dtype=torch.int32, device=DEV) if varlen else None
    r = B.chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0, tok(d),
                    d_fin, cu, n_seq=n_seq)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(r["dS0"], d_fin)
    for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dgate"):
        assert r[n].numel() == 0, n
