"""Brute-force KDA in NumPy with explicit dk x dk transition matrices.

TEST INFRASTRUCTURE ONLY (see the package docstring). Written independently
of ``kda_oracle.c``: where the C code multiplies the update out into a rank-1
correction, this file builds the per-token transition as a full matrix,

    A_t = (I - beta_t k_t k_t^T) Diag(alpha_t),   S_t = A_t S_{t-1} + beta_t k_t v_t^T,
    o_t = gate_t * (scale * S_t^T q_t),

which is the reading of KDA given by the K3 training overview
(zuoshipin.com/article/18261) section 2 "KDA" and the K3 explainer
(devpress.csdn.net/awstech/6a72dc33...) section 2: channel-wise retention,
then a delta-rule corrective write. Only for tiny inputs (T ~ 10^2, d <= 16).
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6


def _norm(x, on):
    x = np.asarray(x, dtype=np.float64)
    if not on:
        return x
    return x / np.sqrt(np.sum(x * x) + L2_EPS)


def transition(k, log_alpha, beta, l2norm=True):
    """A_t = (I - b k k^T) Diag(exp(log_alpha)) for one token (dk x dk)."""
    k = _norm(k, l2norm)
    dk = k.shape[0]
    return (np.eye(dk) - float(beta) * np.outer(k, k)) @ np.diag(
        np.exp(np.asarray(log_alpha, dtype=np.float64)))


def forward(q, k, v, log_alpha, beta, gate=None, S0=None, cu_seqlens=None,
            scale=1.0, l2norm=True):
    q, k, v, la = (np.asarray(a, dtype=np.float64) for a in (q, k, v, log_alpha))
    beta = np.asarray(beta, dtype=np.float64)
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = [0, T] if cu_seqlens is None else list(cu_seqlens)
    out = np.zeros((T, H, dv))
    Sf = np.zeros((len(cu) - 1, H, dk, dv))
    for s in range(len(cu) - 1):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[s, h], dtype=np.float64)
            for t in range(cu[s], cu[s + 1]):
                kn = _norm(k[t, h], l2norm)
                qn = _norm(q[t, h], l2norm)
                A = transition(k[t, h], la[t, h], beta[t, h], l2norm)
                S = A @ S + beta[t, h] * np.outer(kn, v[t, h])
                o = scale * (S.T @ qn)
                if gate is not None:
                    o = o * np.asarray(gate[t, h], dtype=np.float64)
                out[t, h] = o
            Sf[s, h] = S
    return out, Sf


def segment_summary(k, v, log_alpha, beta, cu_segs, l2norm=True):
    """X = A_{end} ... A_{start} (explicit product), Z = state from zero."""
    k, v, la = (np.asarray(a, dtype=np.float64) for a in (k, v, log_alpha))
    beta = np.asarray(beta, dtype=np.float64)
    T, H, dk = k.shape
    dv = v.shape[2]
    n = len(cu_segs) - 1
    X = np.zeros((n, H, dk, dk))
    Z = np.zeros((n, H, dk, dv))
    for s in range(n):
        for h in range(H):
            P = np.eye(dk)
            S = np.zeros((dk, dv))
            for t in range(cu_segs[s], cu_segs[s + 1]):
                A = transition(k[t, h], la[t, h], beta[t, h], l2norm)
                P = A @ P
                S = A @ S + beta[t, h] * np.outer(_norm(k[t, h], l2norm), v[t, h])
            X[s, h] = P
            Z[s, h] = S
    return X, Z
