"""Pins for the backward oracle (oracle/autograd.py), CPU only.

The autograd oracle is trusted only through checks that do not use it to check
itself:
* its forward equals the (separately pinned) C oracle;
* every gradient matches central finite differences, along random directions,
  of L = <dO, o> + <dS_final, S_final> evaluated by the fp64 NumPy brute-force
  oracle (the C oracle reads token inputs as float32, too coarse for a
  finite-difference step);
* closed forms in the degenerate case beta = 0, log_alpha = 0 (memory frozen at
  S0, no L2 norm), where each derivative can be written down by hand.
"""
import numpy as np
import pytest

import oracle
from oracle import autograd as AG
from oracle import brute

CU = [0, 5, 5, 14, 23]  # ragged, with an empty sequence
H, DK, DV = 2, 4, 3


def _f32(a):
    """Values the C oracle sees unchanged (it reads token tensors as float32)."""
    return None if a is None else a.astype(np.float32).astype(np.float64)


def _inputs(seed, T=CU[-1], n_seq=len(CU) - 1, gate=True):
    r = np.random.default_rng(seed)
    x = {
        "q": r.standard_normal((T, H, DK)),
        "k": r.standard_normal((T, H, DK)),
        "v": r.standard_normal((T, H, DV)),
        "log_alpha": -np.exp(r.standard_normal((T, H, DK)) - 1.5),
        "beta": 1.0 / (1.0 + np.exp(-r.standard_normal((T, H)))),
        "gate": (1.0 / (1.0 + np.exp(-r.standard_normal((T, H, DV))))) if gate else None,
        "S0": 0.5 * r.standard_normal((n_seq, H, DK, DV)),
    }
    cot = {"d_out": r.standard_normal((T, H, DV)),
           "d_final": r.standard_normal((n_seq, H, DK, DV))}
    x = {n: (a if n == "S0" else _f32(a)) for n, a in x.items()}
    return x, cot


def _brute_loss(x, cot, scale, l2norm):
    out, sf = brute.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                            x["S0"], CU, scale=scale, l2norm=l2norm)
    return float(np.sum(out * cot["d_out"]) + np.sum(sf * cot["d_final"]))


@pytest.mark.parametrize("l2norm", [True, False])
@pytest.mark.parametrize("gate", [True, False])
def test_forward_matches_c_oracle(l2norm, gate):
    import torch
    x, _ = _inputs(1, gate=gate)
    t = {n: (None if a is None else torch.from_numpy(a)) for n, a in x.items()}
    out, sf = AG.recurrence(t["q"], t["k"], t["v"], t["log_alpha"], t["beta"], t["gate"],
                            t["S0"], CU, scale=0.8, l2norm=l2norm)
    ro, rs = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                            x["S0"], CU, scale=0.8, l2norm=l2norm)
    assert np.max(np.abs(out.numpy() - ro)) <= 1e-12 * max(1.0, np.max(np.abs(ro)))
    assert np.max(np.abs(sf.numpy() - rs)) <= 1e-12 * max(1.0, np.max(np.abs(rs)))


@pytest.mark.parametrize("l2norm", [True, False])
@pytest.mark.parametrize("name", ["q", "k", "v", "log_alpha", "beta", "gate", "S0"])
def test_gradients_match_finite_differences(name, l2norm):
    """<grad_x L, d> against (L(x + e d) - L(x - e d)) / 2e on the brute-force oracle."""
    x, cot = _inputs(2)
    scale = 0.9
    g = AG.backward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"], CU,
                    cot["d_out"], cot["d_final"], scale=scale, l2norm=l2norm)
    r = np.random.default_rng(3)
    for _ in range(3):
        d = r.standard_normal(x[name].shape)
        eps = 1e-5
        xp = dict(x)
        xm = dict(x)
        xp[name] = x[name] + eps * d
        xm[name] = x[name] - eps * d
        fd = (_brute_loss(xp, cot, scale, l2norm) - _brute_loss(xm, cot, scale, l2norm)) / (2 * eps)
        an = float(np.sum(g["d" + name] * d))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_closed_forms_frozen_memory():
    """beta = 0, log_alpha = 0, no L2 norm: S_t = S0 for every t, so with
    w_t = g_t * dO_t and u_t = v_t - S0^T k_t (per head):
      dq_t = scale S0 w_t;  dgate_t = scale dO_t * (S0^T q_t);  dv = 0;  dk = 0;
      dS0 = scale sum_t q_t w_t^T + dS_final;
      dlog_alpha_t = sum_{t' >= t} scale q_t' * (S0 w_t') + diag(S0 dS_final^T);
      dbeta_t = sum_{t' >= t} scale (q_t' . k_t)(w_t' . u_t) + k_t^T dS_final u_t."""
    x, cot = _inputs(4)
    x["beta"][:] = 0.0
    x["log_alpha"][:] = 0.0
    scale = 0.7
    g = AG.backward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"], CU,
                    cot["d_out"], cot["d_final"], scale=scale, l2norm=False)
    for s in range(len(CU) - 1):
        lo, hi = CU[s], CU[s + 1]
        S0, dSf = x["S0"][s], cot["d_final"][s]
        assert np.allclose(g["dS0"][s],
                           dSf + scale * np.einsum("thc,thj->hcj", x["q"][lo:hi],
                                                   x["gate"][lo:hi] * cot["d_out"][lo:hi]),
                           rtol=0, atol=1e-12)
        for t in range(lo, hi):
            w = x["gate"][t] * cot["d_out"][t]                      # [H, dv]
            u = x["v"][t] - np.einsum("hcj,hc->hj", S0, x["k"][t])  # [H, dv]
            assert np.allclose(g["dq"][t], scale * np.einsum("hcj,hj->hc", S0, w), atol=1e-12)
            assert np.allclose(g["dgate"][t],
                               scale * cot["d_out"][t] * np.einsum("hcj,hc->hj", S0, x["q"][t]),
                               atol=1e-12)
            assert np.allclose(g["dv"][t], 0.0, atol=1e-12)
            assert np.allclose(g["dk"][t], 0.0, atol=1e-12)
            dla = np.einsum("hcj,hcj->hc", S0, dSf).copy()
            db = np.einsum("hc,hcj,hj->h", x["k"][t], dSf, u).copy()
            for tp in range(t, hi):
                wp = x["gate"][tp] * cot["d_out"][tp]
                dla += scale * x["q"][tp] * np.einsum("hcj,hj->hc", S0, wp)
                db += scale * np.einsum("hc,hc->h", x["q"][tp], x["k"][t]) * np.einsum(
                    "hj,hj->h", wp, u)
            assert np.allclose(g["dlog_alpha"][t], dla, atol=1e-10)
            assert np.allclose(g["dbeta"][t], db, atol=1e-10)


def test_empty_sequence_passes_final_cotangent_through():
    x, cot = _inputs(5)
    g = AG.backward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"], CU,
                    cot["d_out"], cot["d_final"], scale=1.0)
    assert CU[1] == CU[2]
    assert np.array_equal(g["dS0"][1], cot["d_final"][1])
