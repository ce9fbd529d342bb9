"""kda_segmented_fwd (summaries + ordered scan + segment re-run over one set of update
cards) against the oracle and against the three separate calls (needs a GPU)."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from util import TOL, np32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dk,dv,dtype", [(128, 128, torch.bfloat16), (64, 64, torch.float32)])
def test_segmented_ragged_vs_oracle(dk, dv, dtype):
    """Ragged segments (100, 37, 250, 64, 1 tokens) of one sequence with an initial state:
    the output and final state equal the plain recurrence over the whole sequence, and the
    recovered entry states equal its states at the segment bounds."""
    seg = [100, 37, 250, 64, 1]
    H, T = 2, sum(seg)
    bounds = [0] + np.cumsum(seg).tolist()
    x = inputs.tokens(T, H, dk, dv, dtype, seed=61, device=DEV)
    S0 = inputs.state(1, H, dk, dv, seed=62, device=DEV)[0].contiguous()
    out, fs, ent = B.segmented_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                                   S0, torch.tensor(bounds, dtype=torch.int32, device=DEV),
                                   scale=0.8)
    assert B.kda_get_error() == B.KDA_OK
    args = [np32(x[n]) for n in ("q", "k", "v", "log_alpha", "beta", "gate")]
    s0 = np32(S0).astype(np.float64)[None]
    ro, rs = oracle.forward(*args, s0, [0, T], scale=0.8)
    tol = TOL[dtype]
    assert rel_err(np32(out), ro) <= tol
    assert rel_err(np32(fs), rs[0]) <= tol
    for i, b in enumerate(bounds[:-1]):
        _, re = oracle.forward(*args, s0, [0, T], scale=0.8, t_stop=[b])
        assert rel_err(np32(ent[i]), re[0]) <= tol, i


def test_segmented_longctx_equals_three_calls():
    """1,048,576 tokens x 16 heads in 8 segments: bitwise the same output, final state and
    entry states as kda_segment_summary + kda_scan_combine + kda_chunk_fwd."""
    w = inputs.WORKLOADS["longctx"]
    T, H, n_seg = w.T_total, w.H, w.n_segments
    x = inputs.make(w, device=DEV)
    cu = torch.arange(0, T + 1, T // n_seg, dtype=torch.int32, device=DEV)
    out, fs, ent = B.segmented_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                                   None, cu)
    torch.cuda.synchronize()
    X, Z = B.segment_summary(x["k"], x["v"], x["log_alpha"], x["beta"], cu)
    E, Sf = B.scan_combine(X, Z, None)
    out3, _ = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                          E.contiguous(), cu, n_seq=n_seg, output_final_state=False)
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(ent, E)
    assert torch.equal(fs, Sf)
    assert torch.equal(out, out3)
