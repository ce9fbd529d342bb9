"""Pins for the gate-preparation oracle (oracle/gates.py) and its autograd twin."""
import math

import numpy as np
import pytest

import oracle
from oracle import autograd as AG
from oracle import brute
from oracle import gates


def test_sigmoid_matches_library_and_symmetry():
    special = pytest.importorskip("scipy.special")
    x = np.linspace(-30, 30, 601)
    assert np.allclose(gates.sigmoid(x), special.expit(x), rtol=1e-15, atol=0)
    assert np.allclose(gates.sigmoid(-x), 1.0 - gates.sigmoid(x), atol=1e-15)
    assert gates.sigmoid(0.0) == 0.5


def test_log_alpha_bound_and_shape():
    a_star = math.log(math.log(2.0))          # -e^a = log 1/2 exactly here
    assert math.isclose(gates.log_alpha_of(a_star), math.log(0.5), rel_tol=1e-15)
    assert gates.log_alpha_of(5.0) == math.log(0.5)               # clipped at the bound
    assert math.isclose(gates.log_alpha_of(-3.0), -math.exp(-3.0), rel_tol=1e-15)
    assert -1e-17 < gates.log_alpha_of(-40.0) < 0.0               # retention -> 1
    a = np.linspace(-10, 3, 1001)
    la = gates.log_alpha_of(a)
    assert np.all(np.diff(la) <= 0)                               # monotone non-increasing
    alpha = np.exp(la)
    assert np.all((alpha >= 0.5) & (alpha < 1.0))


def test_autograd_gate_transform_matches_definitions():
    """The autograd oracle with gate_logits equals the C forward oracle fed with the
    prepared gates; its gradients match finite differences of the same composition."""
    import torch
    r = np.random.default_rng(7)
    T, H, dk, dv = 21, 2, 4, 3
    cu = [0, 9, 21]
    raw = {"q": r.standard_normal((T, H, dk)), "k": r.standard_normal((T, H, dk)),
           "v": r.standard_normal((T, H, dv)), "a": r.standard_normal((T, H, dk)) - 1.0,
           "bx": r.standard_normal((T, H)), "gx": r.standard_normal((T, H, dv))}
    raw = {n: x.astype(np.float32).astype(np.float64) for n, x in raw.items()}
    b, g, la = gates.gate_prep(raw["bx"], raw["gx"], raw["a"])
    tb, tg, tla = AG.prepare_gates(torch.from_numpy(raw["bx"]), torch.from_numpy(raw["gx"]),
                                   torch.from_numpy(raw["a"]))
    assert np.allclose(tb.numpy(), b, rtol=1e-15) and np.allclose(tg.numpy(), g, rtol=1e-15)
    assert np.allclose(tla.numpy(), la, rtol=1e-15)
    d_out = r.standard_normal((T, H, dv))

    def loss(bx, gx, a):
        bb, gg, ll = gates.gate_prep(bx, gx, a)
        out, _ = brute.forward(raw["q"], raw["k"], raw["v"], ll, bb, gg, None, cu)
        return float(np.sum(out * d_out))

    grads = AG.backward(raw["q"], raw["k"], raw["v"], raw["a"], raw["bx"], raw["gx"], None, cu,
                        d_out, None, gate_logits=True)
    eps = 1e-6
    for name, key in (("bx", "dbeta"), ("gx", "dgate"), ("a", "dlog_alpha")):
        d = r.standard_normal(raw[name].shape)
        args = {"bx": raw["bx"], "gx": raw["gx"], "a": raw["a"]}
        xp = dict(args, **{name: args[name] + eps * d})
        xm = dict(args, **{name: args[name] - eps * d})
        fd = (loss(**xp) - loss(**xm)) / (2 * eps)
        an = float(np.sum(grads[key] * d))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)
    # and the forward composition equals the C oracle on the prepared gates
    out_c, _ = oracle.forward(raw["q"], raw["k"], raw["v"], la, b, g, None, cu)
    out_b, _ = brute.forward(raw["q"], raw["k"], raw["v"], la, b, g, None, cu)
    assert np.max(np.abs(out_c - out_b)) < 1e-6
