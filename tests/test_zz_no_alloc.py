"""kda_chunk_fwd_noalloc: chunked prefill with the library's fixed device
scratch, for callers that cannot allocate device memory where they run the
mixer (no workspace argument; the library allocates nothing either).

It runs the same kernels on the same schedule as kda_chunk_fwd; only the
scratch address differs. So the two must agree bit for bit, and every case
below is compared with torch.equal: a stale byte left in the shared scratch by
an earlier, larger call would show up as a difference.

Kept in its own file, named to be collected last, so that a run stopping at
the first failure has already run every other test.
"""
import pytest
import torch

from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH = 64 << 20  # the static scratch of kda_chunk_fwd_noalloc, bytes


def _case(seed, lengths, H=4, d=128, dtype=torch.bfloat16):
    T = sum(lengths)
    x = inputs.tokens(T, H, d, d, dtype, seed=seed, device=DEV)
    cu = torch.tensor([0] + list(torch.tensor(lengths).cumsum(0).tolist()), dtype=torch.int32,
                      device=DEV)
    S0 = inputs.state(len(lengths), H, d, d, seed=seed + 1, device=DEV)
    return x, cu, S0


def _run(fn, x, cu, S0, **kw):
    n_seq = cu.numel() - 1
    T, H, d = x["v"].shape
    out = torch.full_like(x["v"], float("nan"))
    fs = torch.full((n_seq, H, d, d), float("nan"), dtype=torch.float32, device=DEV)
    fn(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, S0, fs, cu, n_seq, **kw)
    return out, fs


def _same_as_workspace_entry(x, cu, S0):
    o_ref, s_ref = _run(B.kda_chunk_fwd, x, cu, S0)
    o_na, s_na = _run(B.kda_chunk_fwd_noalloc, x, cu, S0)
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(o_na, o_ref)
    assert torch.equal(s_na, s_ref)


def test_noalloc_matches_workspace_entry_point_twice():
    """Two calls in a row (different inputs and shapes) equal kda_chunk_fwd bit for bit."""
    for seed, lengths in ((300, [200, 77, 64]), (301, [1, 130, 0, 65])):
        x, cu, S0 = _case(seed, lengths)
        _same_as_workspace_entry(x, cu, S0)


def test_noalloc_split_schedule():
    """Few (sequence, head) pairs and long sequences: the split prefill, whose scratch also
    holds the state handed between the two parts."""
    lengths = [2048, 2048]
    n_seq, H = len(lengths), 4
    assert B.kda_chunk_fwd_launches(sum(lengths), n_seq, H, 128, 128, varlen=True) == 5
    x, cu, S0 = _case(303, lengths, H=H)
    _same_as_workspace_entry(x, cu, S0)


def test_noalloc_simt_path():
    """fp32 inputs with dk = dv = 64 take the SIMT kernels and their scratch layout."""
    x, cu, S0 = _case(304, [150, 64, 1], H=3, d=64, dtype=torch.float32)
    _same_as_workspace_entry(x, cu, S0)


def test_noalloc_just_under_the_limit_then_small():
    """The largest single-sequence problem (H = 4, d = 128) whose scratch fits, then a small
    one: the second call must not see the first one's leftovers."""
    H = 4
    T = 64
    while B.kda_chunk_fwd_workspace_size(T + 64, 1, H, 128, 128) <= SCRATCH:
        T += 64
    need = B.kda_chunk_fwd_workspace_size(T, 1, H, 128, 128)
    assert SCRATCH - need < 2 * H * 98816 + 512 * 1024  # within two chunks of the limit
    x, cu, S0 = _case(305, [T], H=H)
    _same_as_workspace_entry(x, cu, S0)
    x, cu, S0 = _case(306, [100, 33], H=H)
    _same_as_workspace_entry(x, cu, S0)


def test_noalloc_rejects_problems_beyond_the_scratch():
    lengths = [4096] * 4
    H, d = 16, 128
    assert B.kda_chunk_fwd_workspace_size(sum(lengths), 4, H, d, d) > SCRATCH
    x, cu, S0 = _case(302, lengths, H=H, d=d)
    with pytest.raises(B.KdaError) as ei:
        _run(B.kda_chunk_fwd_noalloc, x, cu, S0)
    assert ei.value.status == B.KDA_ERR_WORKSPACE
    assert "static scratch" in str(ei.value)
