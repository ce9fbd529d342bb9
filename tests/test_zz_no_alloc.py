"""kda_chunk_fwd_noalloc: chunked prefill with the library's fixed device
scratch, for callers that cannot allocate device memory where they run the
mixer (no workspace argument; the library allocates nothing either).

Kept in its own file, named to be collected last, so that a run stopping at
the first failure has already run every other test.
"""
import pytest
import torch

from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from util import TOL, np32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, lengths, H=4, d=128):
    T = sum(lengths)
    x = inputs.tokens(T, H, d, d, torch.bfloat16, seed=seed, device=DEV)
    cu = torch.tensor([0] + list(torch.tensor(lengths).cumsum(0).tolist()), dtype=torch.int32,
                      device=DEV)
    S0 = inputs.state(len(lengths), H, d, d, seed=seed + 1, device=DEV)
    return x, cu, S0


def _run(fn, x, cu, S0, **kw):
    n_seq = cu.numel() - 1
    T, H, d = x["v"].shape
    out = torch.empty_like(x["v"])
    fs = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=DEV)
    fn(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, S0, fs, cu, n_seq, **kw)
    return out, fs


def test_noalloc_matches_workspace_entry_point_twice():
    """Two calls in a row (different inputs and shapes) agree with kda_chunk_fwd."""
    for seed, lengths in ((300, [200, 77, 64]), (301, [1, 130, 0, 65])):
        x, cu, S0 = _case(seed, lengths)
        o_ref, s_ref = _run(B.kda_chunk_fwd, x, cu, S0)
        o_na, s_na = _run(B.kda_chunk_fwd_noalloc, x, cu, S0)
        assert B.kda_get_error() == B.KDA_OK
        assert rel_err(np32(o_na), np32(o_ref)) <= TOL[torch.bfloat16]
        assert rel_err(np32(s_na), np32(s_ref)) <= TOL[torch.bfloat16]


def test_noalloc_rejects_problems_beyond_the_scratch():
    lengths = [4096] * 4
    H, d = 16, 128
    assert B.kda_chunk_fwd_workspace_size(sum(lengths), 4, H, d, d) > 64 << 20
    x, cu, S0 = _case(302, lengths, H=H, d=d)
    with pytest.raises(B.KdaError) as ei:
        _run(B.kda_chunk_fwd_noalloc, x, cu, S0)
    assert ei.value.status == B.KDA_ERR_WORKSPACE
    assert "static scratch" in str(ei.value)
