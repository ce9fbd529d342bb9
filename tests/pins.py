"""Pins for the KDA oracle: facts fixed by the pages or by mathematics.

Each ``pin_*`` takes an oracle object (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with the fact. They are run against
the real oracle (test_oracle_pins.py) and against deliberately broken builds
of it (test_oracle_mutants.py), which must each fail at least one pin.

Sources for the facts:
  * K3 explainer (devpress.csdn.net/awstech/6a72dc33...), section 2: the
    delta-rule write predicts from memory and stores the error (write-then-read
    returns the written value; a repeated key is overwritten, not summed).
  * K3 training overview (zuoshipin.com/article/18261), section 2 "KDA":
    channel-wise forget gate (per-key-channel decay), output gate.
  * Same page, section 3 "KDA context parallel": two fixed-size summaries per
    segment, merged in order by a prefix scan, recover the exact entry state.
  * Same page, section 4 "FlashKDA" and the K3 explainer's prefix-cache
    section 14: state hand-off, so a run resumed from a stored state equals an
    uninterrupted run.
"""
from __future__ import annotations

import os

import numpy as np

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def rand_case(seed, T, H, dk, dv, n_S0=None, beta=None, log_alpha_lo=np.log(0.5)):
    r = np.random.default_rng(seed)
    f = np.float32
    c = {
        "q": r.standard_normal((T, H, dk)).astype(f),
        "k": r.standard_normal((T, H, dk)).astype(f),
        "v": r.standard_normal((T, H, dv)).astype(f),
        "log_alpha": np.maximum(-np.exp(r.standard_normal((T, H, dk)) - 2.0),
                                log_alpha_lo).astype(f),
        "beta": (1.0 / (1.0 + np.exp(-r.standard_normal((T, H))))).astype(f),
        "gate": (1.0 / (1.0 + np.exp(-r.standard_normal((T, H, dv))))).astype(f),
    }
    if beta is not None:
        c["beta"] = np.full((T, H), beta, dtype=f)
    if n_S0:
        c["S0"] = 0.3 * r.standard_normal((n_S0, H, dk, dv))
    return c


def unit_keys(rng, n, dk):
    """Keys with four entries of +-1/2 and the rest 0: exactly unit length."""
    keys = np.zeros((n, dk), dtype=np.float32)
    for i in range(n):
        idx = rng.choice(dk, 4, replace=False)
        keys[i, idx] = 0.5 * rng.choice([-1.0, 1.0], 4)
    return keys


# --------------------------------------------------------------------------
def pin_brute_force(orc):
    """Rank-1 C recurrence == explicit-matrix NumPy recurrence on tiny cases."""
    cases = [
        dict(seed=1, T=17, H=2, dk=8, dv=4, cu=None, S0=False, l2=True, scale=1.0),
        dict(seed=2, T=20, H=1, dk=4, dv=8, cu=[0, 7, 7, 20], S0=True, l2=True, scale=0.5),
        dict(seed=3, T=9, H=3, dk=8, dv=8, cu=[0, 5, 9], S0=True, l2=False, scale=1.25),
    ]
    for c in cases:
        n_seq = 1 if c["cu"] is None else len(c["cu"]) - 1
        x = rand_case(c["seed"], c["T"], c["H"], c["dk"], c["dv"], n_S0=n_seq if c["S0"] else None)
        args = (x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x.get("S0"), c["cu"])
        o1, s1 = orc.forward(*args, scale=c["scale"], l2norm=c["l2"])
        o2, s2 = brute.forward(*args, scale=c["scale"], l2norm=c["l2"])
        assert rel_err(o1, o2) < 1e-12, ("out", c, rel_err(o1, o2))
        assert rel_err(s1, s2) < 1e-12, ("state", c, rel_err(s1, s2))


def pin_delta_write(orc):
    """beta=1, |k|=1: after the write, S_t^T k_t = v_t exactly, for any decay and history."""
    rng = np.random.default_rng(11)
    T, H, dk, dv = 40, 2, 8, 5
    x = rand_case(12, T, H, dk, dv, n_S0=1, beta=1.0)
    for h in range(H):
        x["k"][:, h] = unit_keys(rng, T, dk)
    x["q"] = x["k"].copy()
    o, _ = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, x["S0"],
                       scale=1.0, l2norm=False)
    assert rel_err(o, x["v"]) < 1e-13, rel_err(o, x["v"])
    # With the library's L2 normalisation the key is k/sqrt(1 + 1e-6): the
    # read-back error is (1 - |k|^2) times the prediction error, about 1e-6.
    o, _ = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, x["S0"],
                       scale=1.0, l2norm=True)
    assert rel_err(o, x["v"]) < 1e-5, rel_err(o, x["v"])


def pin_orthonormal_retrieval(orc):
    """alpha=1, beta=1, orthonormal keys: querying key j returns the last value
    written with key j (zero if none yet)."""
    rng = np.random.default_rng(21)
    T, dk, dv = 30, 4, 3
    basis = 0.5 * np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]],
                           dtype=np.float32)
    wk = rng.integers(0, dk, T)
    qk = rng.integers(0, dk, T)
    v = rng.standard_normal((T, 1, dv)).astype(np.float32)
    k = basis[wk][:, None, :]
    q = basis[qk][:, None, :]
    la = np.zeros((T, 1, dk), dtype=np.float32)
    b = np.ones((T, 1), dtype=np.float32)
    o, _ = orc.forward(q, k, v, la, b, None, None, scale=1.0, l2norm=False)
    last = {}
    for t in range(T):
        last[wk[t]] = v[t, 0]
        want = last.get(qk[t], np.zeros(dv))
        assert np.max(np.abs(o[t, 0] - want)) < 1e-13, (t, o[t, 0], want)


def pin_golden_project_status(orc):
    """The K3 explainer's four-message example (tests/golden fixture)."""
    fx = {}
    with open(os.path.join(GOLDEN, "delta_rule_project_status.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, *vals = line.split()
            fx.setdefault(name, []).append([float(x) for x in vals])
    dk, dv = int(fx["dk"][0][0]), int(fx["dv"][0][0])
    key = np.array(fx["key"][0], dtype=np.float32)
    vals = np.array(fx["value"], dtype=np.float32)
    T = vals.shape[0]
    k = np.tile(key, (T, 1))[:, None, :]
    o, _ = orc.forward(k, k, vals[:, None, :], np.zeros((T, 1, dk), np.float32),
                       np.ones((T, 1), np.float32), None, None, scale=1.0, l2norm=False)
    assert np.array_equal(o[:, 0, :], np.array(fx["expect"])), o[:, 0, :]
    # the same stream through a purely additive memory (beta -> write v, no
    # correction) is what the delta rule avoids; keep the contrast explicit
    assert not np.array_equal(o[-1, 0], np.array(fx["additive_final"][0]))
    assert dv == vals.shape[1]


def pin_beta_zero(orc):
    """beta=0: no write; S_t = Diag(exp(G_t)) S0 and o_t = g * scale * S0^T (exp(G_t) * q_t),
    with G_t the running sum of log_alpha from the start of the sequence."""
    T, H, dk, dv = 25, 2, 8, 6
    cu = [0, 11, 25]
    x = rand_case(31, T, H, dk, dv, n_S0=2, beta=0.0)
    o, S = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"],
                       cu, scale=0.75, l2norm=True)
    for s in range(2):
        for h in range(H):
            G = np.zeros(dk)
            for t in range(cu[s], cu[s + 1]):
                G = G + x["log_alpha"][t, h].astype(np.float64)
                qn = x["q"][t, h].astype(np.float64)
                qn = qn / np.sqrt(np.sum(qn * qn) + 1e-6)
                want = 0.75 * x["gate"][t, h].astype(np.float64) * (x["S0"][s, h].T @ (np.exp(G) * qn))
                assert rel_err(o[t, h], want) < 1e-12
            assert rel_err(S[s, h], np.exp(G)[:, None] * x["S0"][s, h]) < 1e-12


def pin_gla_limit(orc):
    """beta = eps -> 0 from a zero state: o/eps tends to channel-decayed linear
    attention, sum_{i<=t} <q_t * exp(G_t - G_i), k_i> v_i (first order in eps)."""
    eps = 1e-7
    T, H, dk, dv = 48, 1, 8, 4
    x = rand_case(41, T, H, dk, dv, beta=eps)
    o, _ = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, None,
                       scale=1.0, l2norm=True)
    q = x["q"][:, 0].astype(np.float64)
    k = x["k"][:, 0].astype(np.float64)
    q /= np.sqrt(np.sum(q * q, 1, keepdims=True) + 1e-6)
    k /= np.sqrt(np.sum(k * k, 1, keepdims=True) + 1e-6)
    G = np.cumsum(x["log_alpha"][:, 0].astype(np.float64), axis=0)
    beps = float(x["beta"][0, 0])
    want = np.zeros((T, dv))
    for t in range(T):
        for i in range(t + 1):
            want[t] += np.dot(q[t] * np.exp(G[t] - G[i]), k[i]) * x["v"][i, 0]
    assert rel_err(o[:, 0] / beps, want) < 1e-4, rel_err(o[:, 0] / beps, want)


def pin_segment_scan(orc):
    """Segment summaries + ordered scan reproduce the monolithic recurrence:
    entry states, final state; X is the explicit product of transitions and a
    contraction (spectral norm <= 1)."""
    T, H, dk, dv = 40, 2, 8, 6
    cu = [0, 9, 9, 23, 40]
    x = rand_case(51, T, H, dk, dv, n_S0=1)
    X, Z = orc.segment_summary(x["k"], x["v"], x["log_alpha"], x["beta"], cu, l2norm=True)
    Xb, Zb = brute.segment_summary(x["k"], x["v"], x["log_alpha"], x["beta"], cu, l2norm=True)
    assert rel_err(X, Xb) < 1e-12 and rel_err(Z, Zb) < 1e-12
    for s in range(len(cu) - 1):
        for h in range(H):
            assert np.linalg.norm(X[s, h], 2) <= 1.0 + 1e-12
    E, Sf = orc.scan_combine(X, Z, x["S0"][0])
    for s in range(len(cu) - 1):
        _, Sp = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, x["S0"],
                            [0, T], t_stop=[cu[s]], l2norm=True)
        assert rel_err(E[s], Sp[0]) < 1e-12, s
    _, Sm = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, x["S0"],
                        [0, T], l2norm=True)
    assert rel_err(Sf, Sm[0]) < 1e-12
    E0, _ = orc.scan_combine(X, Z, None)
    assert np.all(E0[0] == 0.0)


def pin_resume(orc):
    """Run [0, a) then resume [a, T) from the stored state == one run over [0, T)."""
    T, H, dk, dv, a = 33, 2, 8, 4, 14
    x = rand_case(61, T, H, dk, dv, n_S0=1)
    o, S = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"])
    sl = lambda d, lo, hi: {n: (v[lo:hi] if n != "S0" else v) for n, v in d.items()}
    x1, x2 = sl(x, 0, a), sl(x, a, T)
    o1, S1 = orc.forward(x1["q"], x1["k"], x1["v"], x1["log_alpha"], x1["beta"], x1["gate"],
                         x["S0"])
    o2, S2 = orc.forward(x2["q"], x2["k"], x2["v"], x2["log_alpha"], x2["beta"], x2["gate"], S1)
    assert rel_err(np.concatenate([o1, o2]), o) < 1e-12
    assert rel_err(S2, S) < 1e-12


def pin_decode(orc):
    """decode_step with a slot map == one-token forward per sequence."""
    N, H, dk, dv = 5, 2, 8, 6
    x = rand_case(71, N, H, dk, dv, n_S0=N)
    slot = np.array([3, 0, 4, 1, 2])
    state = np.ascontiguousarray(x["S0"].copy())
    o = orc.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], state,
                        slot, scale=0.9)
    for n in range(N):
        on, Sn = orc.forward(x["q"][n:n + 1], x["k"][n:n + 1], x["v"][n:n + 1],
                             x["log_alpha"][n:n + 1], x["beta"][n:n + 1], x["gate"][n:n + 1],
                             x["S0"][slot[n]:slot[n] + 1], scale=0.9)
        assert rel_err(o[n], on[0]) < 1e-12
        assert rel_err(state[slot[n]], Sn[0]) < 1e-12


def pin_permutation(orc):
    """Value channels are independent: permuting v and gate columns permutes
    o and the state columns; heads are independent."""
    T, H, dk, dv = 21, 3, 8, 7
    x = rand_case(81, T, H, dk, dv, n_S0=1)
    o, S = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"])
    p = np.random.default_rng(82).permutation(dv)
    op, Sp = orc.forward(x["q"], x["k"], x["v"][:, :, p], x["log_alpha"], x["beta"],
                         x["gate"][:, :, p], x["S0"][:, :, :, p])
    assert rel_err(op, o[:, :, p]) < 1e-12 and rel_err(Sp, S[:, :, :, p]) < 1e-12
    hp = np.array([2, 0, 1])
    oh, Sh = orc.forward(x["q"][:, hp], x["k"][:, hp], x["v"][:, hp], x["log_alpha"][:, hp],
                         x["beta"][:, hp], x["gate"][:, hp], x["S0"][:, hp])
    assert rel_err(oh, o[:, hp]) < 1e-12 and rel_err(Sh, S[:, hp]) < 1e-12


def pin_l2norm_invariance(orc):
    """With L2 normalisation on, scaling q and k by positive factors changes
    nothing beyond the 1e-6 eps inside the square root."""
    T, H, dk, dv = 19, 2, 8, 5
    x = rand_case(91, T, H, dk, dv, n_S0=1)
    o, S = orc.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"])
    o2, S2 = orc.forward(8.0 * x["q"], 0.25 * x["k"] * 16.0, x["v"], x["log_alpha"], x["beta"],
                         x["gate"], x["S0"])
    assert rel_err(o2, o) < 1e-6 and rel_err(S2, S) < 1e-6


ALL_PINS = [pin_brute_force, pin_delta_write, pin_orthonormal_retrieval,
            pin_golden_project_status, pin_beta_zero, pin_gla_limit, pin_segment_scan,
            pin_resume, pin_decode, pin_permutation, pin_l2norm_invariance]
