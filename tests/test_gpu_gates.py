"""Fused gate preparation (KDA_GATE_LOGITS) against the oracle (needs a GPU).

The kernels take beta and gate logits and the forget gate's pre-activation a;
the oracle applies oracle/gates.py's definitions in fp64 and runs the plain
recurrence. The pre-activations are drawn so that about one in eight log-retention
values sits on the lower bound log 1/2, so both sides of the clamp are exercised.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from oracle import autograd as AG
from oracle import gates
from util import TOL, np32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _raw(T, H, dk, dv, dtype, seed):
    """Unit-norm-ish q, k and N(0, 1) v from the shared generator; logits drawn here."""
    x = inputs.tokens(T, H, dk, dv, dtype, seed=seed, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    x["log_alpha"] = (torch.randn((T, H, dk), generator=g) - 1.5).to(dtype).to(DEV)
    x["beta"] = torch.randn((T, H), generator=g).to(dtype).to(DEV)
    x["gate"] = torch.randn((T, H, dv), generator=g).to(dtype).to(DEV)
    return x


def _prepared(x):
    b, g, la = gates.gate_prep(np32(x["beta"]), np32(x["gate"]), np32(x["log_alpha"]))
    return b, g, la


@pytest.mark.parametrize("dk,dv,dtype", [(128, 128, torch.bfloat16), (64, 64, torch.float32),
                                         (64, 128, torch.bfloat16)])
def test_forward_with_logits(dk, dv, dtype):
    lengths = [0, 1, 63, 64, 65, 200, 257]
    H = 2
    T = sum(lengths)
    cu = [0] + np.cumsum(lengths).tolist()
    x = _raw(T, H, dk, dv, dtype, 51)
    S0 = inputs.state(len(lengths), H, dk, dv, seed=52, device=DEV)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out, fs = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0, cu_t,
                          scale=0.9, gate_logits=True)
    assert B.kda_get_error() == B.KDA_OK
    b, g, la = _prepared(x)
    assert np.mean(la == np.log(0.5)) > 0.05          # the bound is hit
    ro, rs = oracle.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), la, b, g,
                            np32(S0).astype(np.float64), cu, scale=0.9)
    assert rel_err(np32(out), ro) <= TOL[dtype]
    assert rel_err(np32(fs), rs) <= TOL[dtype]


def test_decode_with_logits():
    N, H, d = 64, 4, 128
    S = inputs.state(N, H, d, d, seed=53, device=DEV).contiguous()
    ref_state = np32(S).astype(np.float64)
    x = _raw(N, H, d, d, torch.bfloat16, 54)
    o = B.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S,
                      gate_logits=True)
    assert B.kda_get_error() == B.KDA_OK
    b, g, la = _prepared(x)
    ro = oracle.decode_step(np32(x["q"]), np32(x["k"]), np32(x["v"]), la, b, g, ref_state)
    assert rel_err(np32(o), ro) <= TOL[torch.bfloat16]
    assert rel_err(np32(S), ref_state) <= TOL[torch.bfloat16]


def test_segment_summary_with_logits():
    lengths = [130, 64, 7]
    T, H, d = sum(lengths), 2, 128
    cu = [0] + np.cumsum(lengths).tolist()
    x = _raw(T, H, d, d, torch.bfloat16, 55)
    X, Z = B.segment_summary(x["k"], x["v"], x["log_alpha"], x["beta"],
                             torch.tensor(cu, dtype=torch.int32, device=DEV), gate_logits=True)
    assert B.kda_get_error() == B.KDA_OK
    b, _, la = _prepared(x)
    rX, rZ = oracle.segment_summary(np32(x["k"]), np32(x["v"]), la, b, cu)
    assert rel_err(np32(X), rX) <= TOL[torch.bfloat16]
    assert rel_err(np32(Z), rZ) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("dk,dv,dtype", [(128, 128, torch.bfloat16), (64, 64, torch.float32)])
def test_backward_with_logits(dk, dv, dtype):
    lengths = [65, 1, 130]
    H = 2
    T = sum(lengths)
    cu = [0] + np.cumsum(lengths).tolist()
    x = _raw(T, H, dk, dv, dtype, 56)
    S0 = inputs.state(len(lengths), H, dk, dv, seed=57, device=DEV)
    gcpu = torch.Generator(device="cpu").manual_seed(58)
    d_out = torch.randn((T, H, dv), generator=gcpu).to(dtype).to(DEV)
    d_fin = torch.randn((len(lengths), H, dk, dv), generator=gcpu).to(DEV)
    got = B.chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0, d_out,
                      d_fin, torch.tensor(cu, dtype=torch.int32, device=DEV), scale=0.9,
                      gate_logits=True)
    assert B.kda_get_error() == B.KDA_OK
    ref = AG.backward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                      np32(x["beta"]), np32(x["gate"]), np32(S0), cu, np32(d_out), np32(d_fin),
                      scale=0.9, gate_logits=True)
    for n in ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dgate", "dS0"):
        e = rel_err(np32(got[n]), ref[n])
        assert e <= TOL[dtype], (n, e)
    # on the bound the retention does not depend on a: its gradient is exactly zero
    on_bound = torch.from_numpy(_prepared(x)[2] == np.log(0.5)).to(DEV)
    assert torch.count_nonzero(got["dlog_alpha"][on_bound]) == 0
