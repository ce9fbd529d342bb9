"""kda_chunk_fwd_host (page-locked host buffers in and out, copies overlapped with the compute
per sequence, the last sequence in time slices) gives bitwise the results of kda_chunk_fwd on
the same values in device memory (needs a GPU)."""
import pytest
import torch

from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs

pytestmark = pytest.mark.gpu

_TOKEN = ("q", "k", "v", "log_alpha", "beta", "gate")


def _device_call(x, S0, n_seq):
    out, fs = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0, None,
                          n_seq=n_seq)
    torch.cuda.synchronize()
    return out.cpu(), fs.cpu()


def _host_call(x, S0, n_seq, tail_slices, flags=B.KDA_QK_L2NORM, with_final=True, buf=None):
    h = {n: (x[n].cpu().pin_memory() if x[n] is not None else None) for n in _TOKEN}
    s0 = S0.cpu().pin_memory() if S0 is not None else None
    T, H, dv = x["v"].shape
    dk = x["k"].shape[-1]
    out = torch.full((T, H, dv), 7.0, dtype=x["v"].dtype).pin_memory()
    fs = torch.full((n_seq, H, dk, dv), 7.0).pin_memory() if with_final else None
    B.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], h["gate"], out, s0,
                         fs, n_seq, flags=flags, tail_slices=tail_slices, device_buffer=buf)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    return out, fs


@pytest.mark.parametrize("tail_slices", [1, 4])
def test_prefill_workload_bitwise(tail_slices):
    """4 x 4096 tokens x 16 heads, bf16, d = 128 (what the end-to-end bench line runs)."""
    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device="cuda")
    n_seq = len(w.lengths)
    out_d, fs_d = _device_call(x, x["S0"], n_seq)
    out_h, fs_h = _host_call(x, x["S0"], n_seq, tail_slices)
    assert torch.equal(out_h, out_d)
    assert torch.equal(fs_h, fs_d)


@pytest.mark.parametrize("n_seq,L,H,d,dtype,tail_slices", [
    (3, 77, 5, 64, torch.float32, 1),       # lengths off the chunk grid, odd head count
    (2, 1100, 4, 128, torch.bfloat16, 1),   # a partial last chunk, tensor-core path
    (2, 1024, 4, 128, torch.bfloat16, 8),   # 8 slices of 128 tokens
    (1, 512, 3, 64, torch.bfloat16, 2),     # one sequence, only slices
])
def test_shapes_bitwise(n_seq, L, H, d, dtype, tail_slices):
    x = inputs.tokens(n_seq * L, H, d, d, dtype, seed=500 + L, device="cuda")
    S0 = inputs.state(n_seq, H, d, d, seed=501 + L, device="cuda")
    out_d, fs_d = _device_call(x, S0, n_seq)
    out_h, fs_h = _host_call(x, S0, n_seq, tail_slices)
    assert torch.equal(out_h, out_d)
    assert torch.equal(fs_h, fs_d)


def test_no_gate_no_states_and_repeat():
    """gate, initial and final state absent; a second call into the same device buffer gives
    the same bits."""
    n_seq, L, H, d = 2, 640, 4, 128
    x = inputs.tokens(n_seq * L, H, d, d, torch.bfloat16, seed=77, device="cuda", with_gate=False)
    out_d, _ = _device_call(x, None, n_seq)
    need = B.kda_chunk_fwd_host_buffer_size(n_seq * L, n_seq, H, d, d, tail_slices=2)
    buf = torch.empty(need, dtype=torch.uint8, device="cuda")
    out1, _ = _host_call(x, None, n_seq, 2, with_final=False, buf=buf)
    out2, _ = _host_call(x, None, n_seq, 2, with_final=False, buf=buf)
    assert torch.equal(out1, out_d)
    assert torch.equal(out2, out_d)


def test_empty_sequences_keep_the_initial_state():
    H, d = 2, 64
    S0 = inputs.state(3, H, d, d, seed=9).pin_memory()
    fs = torch.zeros((3, H, d, d)).pin_memory()
    e = torch.empty((0, H, d), dtype=torch.bfloat16).pin_memory()
    eb = torch.empty((0, H), dtype=torch.bfloat16).pin_memory()
    B.kda_chunk_fwd_host(e, e, e, e, eb, None, e, S0, fs, 3)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(fs, S0)


def test_pageable_memory_is_rejected():
    n_seq, L, H, d = 1, 128, 2, 64
    x = inputs.tokens(n_seq * L, H, d, d, torch.bfloat16, seed=3)  # ordinary (pageable) memory
    out = torch.empty((L, H, d), dtype=torch.bfloat16)
    with pytest.raises(B.KdaError) as ei:
        B.kda_chunk_fwd_host(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out,
                             None, None, n_seq)
    assert ei.value.status == B.KDA_ERR_INVALID_ARG
    assert "page-locked" in str(ei.value)


def _fuzz_fixed_cases():
    import os
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    from test_gpu_fuzz import _draw
    return [i for i in range(48) if _draw(i)[1]]


@pytest.mark.parametrize("i", _fuzz_fixed_cases())
def test_fuzz_fixed_lengths_bitwise(i):
    """The fixed-length cases of the seeded fuzz generator (every head-dim pair, fp32 and bf16,
    with and without gate and initial state): each sequence computed on its own, the last one
    in time slices where its length allows, equals the batch computed in one device call."""
    from test_gpu_fuzz import _draw
    lengths, fixed, H, dk, dv, dtype, scale, gate, l2norm, with_init = _draw(i)
    n_seq, L = len(lengths), lengths[0]
    x = inputs.tokens(n_seq * L, H, dk, dv, dtype, seed=9100 + i, device="cuda", with_gate=gate)
    S0 = inputs.state(n_seq, H, dk, dv, seed=9200 + i, device="cuda") if with_init else None
    flags = B.KDA_QK_L2NORM if l2norm else 0
    out_d, fs_d = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0,
                              None, n_seq=n_seq, scale=scale, l2norm=l2norm)
    torch.cuda.synchronize()
    tail = next((t for t in (4, 2) if L % (64 * t) == 0), 1)
    h = {n: (x[n].cpu().pin_memory() if x[n] is not None else None) for n in _TOKEN}
    out_h = torch.empty((n_seq * L, H, dv), dtype=dtype).pin_memory()
    fs_h = torch.empty((n_seq, H, dk, dv)).pin_memory()
    B.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], h["gate"], out_h,
                         S0.cpu().pin_memory() if S0 is not None else None, fs_h, n_seq,
                         scale=scale, flags=flags, tail_slices=tail)
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(fs_h, fs_d.cpu())
