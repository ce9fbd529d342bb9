"""HostPipeline (copy in / compute / copy out per sequence group on three streams, optionally
per time slice of each sequence or of the last one) gives bitwise the results of one kda_chunk_fwd call on the
device-resident batch (needs a GPU)."""
import pytest
import torch

from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from linear_attention_05_gb300.pipeline import HostPipeline

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("groups,parts,tail_parts", [(4, 1, None), (2, 1, None), (4, 4, None),
                                                    (4, 2, None), (4, 1, 2), (4, 1, 4)])
def test_pipeline_equals_device_call(groups, parts, tail_parts):
    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device="cuda")
    n_seq, L, H, d = len(w.lengths), w.lengths[0], w.H, w.dk
    out_d, fs_d = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                              x["S0"], None, n_seq=n_seq)
    host = {k: v.cpu().pin_memory() for k, v in x.items() if k != "cu_seqlens" and v is not None}
    out_h = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
    fs_h = torch.empty(fs_d.shape, dtype=fs_d.dtype).pin_memory()
    pl = HostPipeline(n_seq, L, H, d, d, dtype=torch.bfloat16, device="cuda", groups=groups,
                      parts=parts, tail_parts=tail_parts)
    pl.run(host, out_h, fs_h)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(fs_h, fs_d.cpu())
