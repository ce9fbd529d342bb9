"""Gate preparation, written out in fp64 (test infrastructure, like the rest of
this package; the library never imports it).

K3 training overview (zuoshipin.com/article/18261) section 2 "KDA": KDA has a
channel-wise forget gate whose per-step retention has a lower bound, and an
output gate; section 4 "FlashKDA" lists the forget gate among the parts of the
per-chunk update card. The pages give no formulas. The readings used here are
the transforms of the synthetic input recipe:
    beta  = sigmoid(beta_logit)                 (write strength in (0, 1))
    g     = sigmoid(gate_logit)                 (sigmoid output gate)
    log_alpha = max(-exp(a), log(1/2))          (retention alpha in [1/2, 1))
"""
from __future__ import annotations

import math

import numpy as np

LOG_HALF = math.log(0.5)


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def log_alpha_of(a):
    a = np.asarray(a, dtype=np.float64)
    return np.maximum(-np.exp(a), LOG_HALF)


def gate_prep(beta_logit=None, gate_logit=None, alpha_logit=None):
    """(beta, g, log_alpha) from their logits / pre-activation; None passes through."""
    return (None if beta_logit is None else sigmoid(beta_logit),
            None if gate_logit is None else sigmoid(gate_logit),
            None if alpha_logit is None else log_alpha_of(alpha_logit))
