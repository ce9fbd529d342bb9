"""A bounded device wait that runs out, on the GPU, without a fault (needs a GPU).

Every wait of the chunked kernels on a bulk copy or on the tensor cores is bounded: when the
limit runs out the kernel records KDA_ERR_TIMEOUT in the device error word and returns
normally, so the context stays usable. kda_selftest_wait_timeout makes such a wait run out on
purpose: one CTA waits on an mbarrier that nothing ever arrives on (no copy and no MMA is in
flight), for a limit of about a millisecond.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from util import TOL, check, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_runs_out_and_reports_timeout():
    assert B.kda_get_error() == B.KDA_OK  # start from a clear word
    st = B.kda_selftest_wait_timeout(1000)
    assert st == B.KDA_OK
    assert B.kda_get_error() == B.KDA_ERR_TIMEOUT
    assert "bounded device wait" in B.kda_last_error_string()
    assert B.kda_get_error() == B.KDA_OK  # the word is cleared on read


def test_normal_call_after_timeout_is_correct():
    B.kda_selftest_wait_timeout(500)
    assert B.kda_get_error() == B.KDA_ERR_TIMEOUT
    lengths = [200, 77]
    cu = [0, 200, 277]
    x = inputs.tokens(sum(lengths), 2, 128, 128, torch.bfloat16, seed=500, device=DEV)
    S0 = inputs.state(2, 2, 128, 128, seed=501, device=DEV)
    out, fs = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0,
                          torch.tensor(cu, dtype=torch.int32, device=DEV), n_seq=2)
    assert B.kda_get_error() == B.KDA_OK
    ro, rs = oracle.forward(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                            np32(x["beta"]), np32(x["gate"]), np32(S0).astype(np.float64), cu)
    check("after_timeout/out_vs_oracle", np32(out), ro, TOL[torch.bfloat16])
    check("after_timeout/state_vs_oracle", np32(fs), rs, TOL[torch.bfloat16])
