"""Gradients of KDA by fp64 autograd of the token recurrence (backward oracle).

TEST INFRASTRUCTURE ONLY, like the rest of this package: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it, and it imports nothing from the library.

What it computes: the derivatives of the scalar
    L = sum_t <dO_t, o_t> + sum_s <dS_final_s, S_final_s>
with respect to q, k, v, log_alpha, beta, gate and the initial state, i.e. the
vector-Jacobian product of the forward pass with cotangents (dO, dS_final).
The forward is written once more, here in PyTorch (fp64, CPU), token by token:
    S' = Diag(exp(log_alpha_t)) S;  u = v_t - S'^T k_t;  S = S' + beta_t k_t u^T;
    o_t = g_t * scale * S^T q_t
(q_t, k_t L2-normalised first when asked: x / sqrt(sum x^2 + 1e-6)). This is the
multiplied-out form of S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T from K3
training overview (zuoshipin.com/article/18261) section 2 "KDA", K3 explainer
(devpress.csdn.net/awstech/6a72dc33...) section 2. Training needs these
gradients: section 4 "FlashKDA" of the training overview presents the chunked
kernel as a training kernel. The derivatives come from torch.autograd; nothing
here is hand-differentiated. The tests pin the forward to the C oracle and the
gradients to central finite differences of the fp64 brute-force oracle.
"""
from __future__ import annotations

import numpy as np
import torch

L2_EPS = 1e-6


def _t(x):
    return torch.tensor(np.asarray(x, dtype=np.float64), dtype=torch.float64, requires_grad=True)


def recurrence(q, k, v, log_alpha, beta, gate, S0, cu_seqlens, scale=1.0, l2norm=True):
    """Differentiable fp64 forward on torch tensors.

    q, k, log_alpha: [T, H, dk]; v, gate: [T, H, dv] (gate may be None); beta: [T, H];
    S0: [n_seq, H, dk, dv] or None. Returns (out [T, H, dv], S_final [n_seq, H, dk, dv])."""
    T, H, dk = k.shape
    dv = v.shape[-1]
    n_seq = len(cu_seqlens) - 1
    outs = []
    finals = []
    for s in range(n_seq):
        S = S0[s] if S0 is not None else torch.zeros((H, dk, dv), dtype=torch.float64)
        for t in range(int(cu_seqlens[s]), int(cu_seqlens[s + 1])):
            kt, qt = k[t], q[t]
            if l2norm:
                kt = kt / torch.sqrt((kt * kt).sum(-1, keepdim=True) + L2_EPS)
                qt = qt / torch.sqrt((qt * qt).sum(-1, keepdim=True) + L2_EPS)
            Sp = torch.exp(log_alpha[t])[:, :, None] * S
            u = v[t] - torch.einsum("hc,hcj->hj", kt, Sp)
            S = Sp + beta[t][:, None, None] * kt[:, :, None] * u[:, None, :]
            o = scale * torch.einsum("hcj,hc->hj", S, qt)
            outs.append(o if gate is None else gate[t] * o)
        finals.append(S)
    out = torch.stack(outs) if outs else torch.zeros((0, H, dv), dtype=torch.float64)
    return out, torch.stack(finals)


def prepare_gates(beta, gate, log_alpha):
    """Differentiable beta = sigmoid(x), g = sigmoid(y), log_alpha = max(-e^a, log 1/2)
    (the definitions of oracle/gates.py) on torch tensors."""
    la = torch.maximum(-torch.exp(log_alpha), torch.tensor(np.log(0.5), dtype=torch.float64))
    return torch.sigmoid(beta), None if gate is None else torch.sigmoid(gate), la


def backward(q, k, v, log_alpha, beta, gate, S0, cu_seqlens, d_out, d_final=None, scale=1.0,
             l2norm=True, gate_logits=False):
    """Vector-Jacobian product of the forward with cotangents (d_out, d_final).

    Arrays in, float64 numpy arrays out: dict with dq, dk, dv, dlog_alpha, dbeta, dgate
    (None when gate is None) and dS0 (gradient of the initial state; zero-state runs
    report the gradient at S0 = 0). gate_logits: beta, gate and log_alpha hold logits and
    the forget gate's pre-activation (prepare_gates), and the gradients are theirs."""
    n_seq = len(cu_seqlens) - 1
    T, H, dk = np.shape(k)
    dv = np.shape(v)[-1]
    xs = {"q": _t(q), "k": _t(k), "v": _t(v), "log_alpha": _t(log_alpha), "beta": _t(beta)}
    xs["gate"] = None if gate is None else _t(gate)
    xs["S0"] = _t(np.zeros((n_seq, H, dk, dv)) if S0 is None else S0)
    b, g, la = xs["beta"], xs["gate"], xs["log_alpha"]
    if gate_logits:
        b, g, la = prepare_gates(b, g, la)
    out, Sf = recurrence(xs["q"], xs["k"], xs["v"], la, b, g, xs["S0"], cu_seqlens, scale=scale,
                         l2norm=l2norm)
    L = (out * torch.as_tensor(np.asarray(d_out, dtype=np.float64))).sum()
    if d_final is not None:
        L = L + (Sf * torch.as_tensor(np.asarray(d_final, dtype=np.float64))).sum()
    names = [n for n in ("q", "k", "v", "log_alpha", "beta", "gate", "S0") if xs[n] is not None]
    if L.requires_grad:
        grads = torch.autograd.grad(L, [xs[n] for n in names], allow_unused=True)
    else:  # no tokens and no final-state cotangent
        grads = [None] * len(names)
    res = {}
    for n, g in zip(names, grads):
        res["d" + n] = (np.zeros(xs[n].shape) if g is None else g.detach().numpy())
    res.setdefault("dgate", None)
    return res
