"""CUDA path vs the fp64 oracle on seeded inputs (needs a GPU).

Metric: max|gpu - ref| / max|ref| per output tensor (o and states separately);
fp32 inputs <= 1e-4, bf16 inputs with fp32 state <= 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from util import TOL, check, np32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_oracle(x, cu, heads=None, scale=1.0, l2norm=True, S0=None, t_stop=None):
    """Oracle on (optionally) a subset of heads."""
    sel = (lambda t: t) if heads is None else (lambda t: t[:, heads])
    g = None if x["gate"] is None else np32(sel(x["gate"]))
    s0 = None
    if S0 is not None:
        s0 = np32(S0 if heads is None else S0[:, heads]).astype(np.float64)
    return oracle.forward(np32(sel(x["q"])), np32(sel(x["k"])), np32(sel(x["v"])),
                          np32(sel(x["log_alpha"])), np32(sel(x["beta"])), g, s0,
                          list(cu), scale=scale, l2norm=l2norm, t_stop=t_stop)


def gpu_chunk(x, cu_list, S0=None, scale=1.0, l2norm=True, fixed=False, gate=True):
    cu = None if fixed else torch.tensor(cu_list, dtype=torch.int32, device=DEV)
    n_seq = len(cu_list) - 1
    out, fs = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                          x["gate"] if gate else None, S0, cu, n_seq=n_seq, scale=scale,
                          l2norm=l2norm)
    assert B.kda_get_error() == B.KDA_OK
    return out, fs


def make_tokens(lengths, H, dk, dv, dtype, seed):
    T = int(sum(lengths))
    x = inputs.tokens(T, H, dk, dv, dtype, seed, device=DEV)
    cu = [0] + list(np.cumsum(lengths).tolist())
    return x, cu


# ---------------------------------------------------------------- the five workloads
def test_tiny_fp32_workload():
    w = inputs.WORKLOADS["tiny"]
    x = inputs.make(w, device=DEV)
    out, fs = gpu_chunk(x, w.cu_seqlens)
    ro, rs = run_oracle(x, w.cu_seqlens)
    check("tiny/out", np32(out), ro, 1e-4)
    check("tiny/state", np32(fs), rs, 1e-4)


def test_prefill_workload_full():
    """4 x 4096 tokens, 16 heads, d=128, bf16, S0 ~ N(0, 0.01): every output."""
    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device=DEV)
    out, fs = gpu_chunk(x, w.cu_seqlens, S0=x["S0"], fixed=True)
    ro, rs = run_oracle(x, w.cu_seqlens, S0=x["S0"])
    check("prefill/out", np32(out), ro, TOL[torch.bfloat16])
    check("prefill/state", np32(fs), rs, TOL[torch.bfloat16])


def test_varlen_workload_sampled_heads():
    """8 packed sequences (~112K tokens), 32 heads: all GPU outputs computed,
    oracle on 3 of the 32 heads (the heads are independent)."""
    w = inputs.WORKLOADS["varlen"]
    x = inputs.make(w, device=DEV)
    out, fs = gpu_chunk(x, w.cu_seqlens)
    heads = [0, 13, 31]
    ro, rs = run_oracle(x, w.cu_seqlens, heads=heads)
    check("varlen/out_heads_0_13_31", np32(out[:, heads]), ro, TOL[torch.bfloat16])
    check("varlen/state_heads_0_13_31", np32(fs[:, heads]), rs, TOL[torch.bfloat16])
    assert torch.isfinite(out).all()


def test_longctx_segment_scan():
    """1,048,576 tokens, 16 heads, 8 segments: summaries + scan + segment
    re-run equal the monolithic chunked pass; the state entering segment 1 and
    a 4096-token slice straddling the segment boundary match the oracle."""
    w = inputs.WORKLOADS["longctx"]
    T, H = w.T_total, w.H
    x = inputs.make(w, device=DEV)
    n_seg = w.n_segments
    L = T // n_seg
    cu_segs = torch.arange(0, T + 1, L, dtype=torch.int32, device=DEV)
    X, Z = B.segment_summary(x["k"], x["v"], x["log_alpha"], x["beta"], cu_segs)
    E, Sf = B.scan_combine(X, Z, None)
    out_seg, fs_seg = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                                  E.contiguous(), cu_segs, n_seq=n_seg)
    out_mono, fs_mono = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                    x["gate"], None, None, n_seq=1)
    assert B.kda_get_error() == B.KDA_OK
    # segmented (scan) path == monolithic path
    check("longctx/final_segmented_vs_monolithic", np32(fs_seg[-1]), np32(fs_mono[0]),
          TOL[torch.bfloat16])
    check("longctx/scan_final_vs_monolithic", np32(Sf), np32(fs_mono[0]), TOL[torch.bfloat16])
    o1 = out_seg[L - 2048:L + 2048].float()
    o2 = out_mono[L - 2048:L + 2048].float()
    check("longctx/slice_segmented_vs_monolithic", o1.cpu().numpy(), o2.cpu().numpy(),
          TOL[torch.bfloat16])
    # oracle on 4 heads, tokens [0, L + 2048): entry state of segment 1 and the slice
    heads = [0, 5, 10, 15]
    t_end = L + 2048
    xs = {k: (v[:t_end] if v is not None and k != "S0" else v) for k, v in x.items()}
    ro, _ = run_oracle(xs, [0, t_end], heads=heads)
    _, rE1 = run_oracle(xs, [0, t_end], heads=heads, t_stop=[L])
    check("longctx/entry_state_segment1_vs_oracle", np32(E[1][heads]), rE1[0],
          TOL[torch.bfloat16])
    sl = slice(L - 2048, L + 2048)
    check("longctx/slice_segmented_vs_oracle", np32(out_seg[sl][:, heads]), ro[sl],
          TOL[torch.bfloat16])
    check("longctx/slice_monolithic_vs_oracle", np32(out_mono[sl][:, heads]), ro[sl],
          TOL[torch.bfloat16])


def test_decode_workload_64_steps():
    """256 sequences x 32 heads, d=128, fp32 states in HBM, 64 steps with fresh
    inputs; every output and the final states vs the oracle."""
    w = inputs.WORKLOADS["decode"]
    N, H, d = len(w.lengths), w.H, w.dk
    S = inputs.state(N, H, d, d, w.seed, device=DEV).contiguous()
    ref_state = np32(S).astype(np.float64)
    worst = 0.0
    for step in range(w.steps):
        x = inputs.tokens(N, H, d, d, w.dtype, w.seed, step=step, device=DEV)
        o = B.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S)
        ro = oracle.decode_step(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                                np32(x["beta"]), np32(x["gate"]), ref_state)
        worst = max(worst, rel_err(np32(o), ro))
    assert B.kda_get_error() == B.KDA_OK
    print(f"PARITY decode/out_worst_step err={worst:.3e} tol=2e-02 "
          f"margin={TOL[torch.bfloat16] / max(worst, 1e-300):.1f}x", flush=True)
    assert worst <= TOL[torch.bfloat16], worst
    check("decode/state_after_64_steps", np32(S), ref_state, TOL[torch.bfloat16])


# ---------------------------------------------------------------- edge cases and shapes
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_varlen_shapes(dk, dv, dtype):
    """Lengths that hit every tail case: empty, 1, 63, 64, 65, 130, 200."""
    lengths = [65, 0, 1, 63, 64, 130, 200]
    x, cu = make_tokens(lengths, 3, dk, dv, dtype, seed=100 + dk + dv)
    S0 = inputs.state(len(lengths), 3, dk, dv, seed=7, device=DEV)
    out, fs = gpu_chunk(x, cu, S0=S0, scale=0.8)
    ro, rs = run_oracle(x, cu, S0=S0, scale=0.8)
    check(f"ragged/{dk}x{dv}/{str(dtype)[6:]}/out", np32(out), ro, TOL[dtype])
    check(f"ragged/{dk}x{dv}/{str(dtype)[6:]}/state", np32(fs), rs, TOL[dtype])
    # the empty sequence hands its initial state through unchanged
    assert torch.equal(fs[1], S0[1])


def test_no_gate_no_l2norm_fp32():
    x, cu = make_tokens([150, 77], 2, 64, 64, torch.float32, seed=5)
    out, fs = gpu_chunk(x, cu, l2norm=False, gate=False)
    x2 = dict(x, gate=None)
    ro, rs = run_oracle(x2, cu, l2norm=False)
    assert rel_err(np32(out), ro) <= 1e-4 and rel_err(np32(fs), rs) <= 1e-4


def test_empty_batch():
    x, cu = make_tokens([0, 0], 2, 128, 128, torch.bfloat16, seed=6)
    S0 = inputs.state(2, 2, 128, 128, seed=6, device=DEV)
    out, fs = gpu_chunk(x, cu, S0=S0)
    assert out.numel() == 0 and torch.equal(fs, S0)


def test_resume_equals_single_pass():
    """Prefix-cache hand-off: run [0, a), resume [a, T) from the stored state."""
    T, a = 640, 320
    x, _ = make_tokens([T], 4, 128, 128, torch.bfloat16, seed=8)
    out, fs = gpu_chunk(x, [0, T])
    x1 = {k: v[:a] for k, v in x.items()}
    x2 = {k: v[a:] for k, v in x.items()}
    o1, s1 = gpu_chunk(x1, [0, a])
    o2, s2 = gpu_chunk(x2, [0, T - a], S0=s1)
    got = torch.cat([o1, o2]).float().cpu().numpy()
    assert rel_err(got, np32(out)) <= 1e-2
    assert rel_err(np32(s2), np32(fs)) <= 1e-2


def test_deterministic():
    x, cu = make_tokens([300, 1000], 4, 128, 128, torch.bfloat16, seed=9)
    o1, s1 = gpu_chunk(x, cu)
    o2, s2 = gpu_chunk(x, cu)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_lower_bound_retention_is_finite():
    """log_alpha at the documented floor on every channel: chunk factors up to
    2^64 stay finite and the result still matches the oracle."""
    x, cu = make_tokens([256], 2, 128, 128, torch.bfloat16, seed=10)
    x["log_alpha"].fill_(-0.6953125)
    out, fs = gpu_chunk(x, cu)
    assert torch.isfinite(out).all() and torch.isfinite(fs).all()
    ro, rs = run_oracle(x, cu)
    assert rel_err(np32(out), ro) <= 2e-2 and rel_err(np32(fs), rs) <= 2e-2


def test_debug_check_reports_precondition():
    x, cu = make_tokens([100], 2, 64, 64, torch.bfloat16, seed=11)
    x["log_alpha"][5, 1, 3] = -2.0
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out = torch.empty_like(x["v"])
    B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, None,
                    None, cu_t, 1, flags=B.KDA_QK_L2NORM | B.KDA_DEBUG_CHECK)
    assert B.kda_get_error() == B.KDA_ERR_PRECONDITION
    assert B.kda_get_error() == B.KDA_OK  # the word is cleared on read


def test_malformed_cu_seqlens_reported():
    x, _ = make_tokens([128], 2, 64, 64, torch.bfloat16, seed=12)
    bad = torch.tensor([0, 100, 50, 128], dtype=torch.int32, device=DEV)  # decreasing
    out = torch.zeros_like(x["v"])
    B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, None,
                    None, bad, 3)
    assert B.kda_get_error() == B.KDA_ERR_INVALID_ARG
    assert not out.any()  # nothing written


# ---------------------------------------------------------------- decode specifics
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_decode_slots_and_shapes(dk, dv):
    N, H, n_slots = 6, 3, 9
    x = inputs.tokens(N, H, dk, dv, torch.float32, seed=20, device=DEV)
    S = inputs.state(n_slots, H, dk, dv, seed=21, device=DEV).contiguous()
    slot = torch.tensor([8, 0, 3, 5, 1, 7], dtype=torch.int32, device=DEV)
    ref = np32(S).astype(np.float64)
    o = B.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S, slot,
                      scale=1.3)
    ro = oracle.decode_step(np32(x["q"]), np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                            np32(x["beta"]), np32(x["gate"]), ref, slot.cpu().numpy(), scale=1.3)
    assert rel_err(np32(o), ro) <= 1e-4
    assert rel_err(np32(S), ref) <= 1e-4  # untouched slots stay equal too


def test_decode_equals_chunk_one_token():
    N, H, d = 4, 2, 128
    x = inputs.tokens(N, H, d, d, torch.bfloat16, seed=30, device=DEV)
    S = inputs.state(N, H, d, d, seed=31, device=DEV).contiguous()
    S_in = S.clone()
    o = B.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S)
    cu = torch.arange(N + 1, dtype=torch.int32, device=DEV)
    oc, sc = B.chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S_in, cu,
                         n_seq=N)
    # bf16 inputs: both paths within the bf16 tolerance of each other (the chunked
    # tensor-core path multiplies bf16-rounded state operands)
    assert rel_err(np32(o), np32(oc)) <= TOL[torch.bfloat16]
    assert rel_err(np32(S), np32(sc)) <= TOL[torch.bfloat16]


def test_decode_bad_slot_reported():
    x = inputs.tokens(2, 1, 64, 64, torch.float32, seed=40, device=DEV)
    S = torch.zeros((2, 1, 64, 64), device=DEV)
    slot = torch.tensor([0, 5], dtype=torch.int32, device=DEV)
    B.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S, slot)
    assert B.kda_get_error() == B.KDA_ERR_INVALID_ARG


# ---------------------------------------------------------------- segment scan specifics
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_segment_summary_vs_oracle(dtype):
    lengths = [100, 0, 64, 257]
    x, cu = make_tokens(lengths, 2, 64, 64, dtype, seed=50)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    X, Z = B.segment_summary(x["k"], x["v"], x["log_alpha"], x["beta"], cu_t)
    assert B.kda_get_error() == B.KDA_OK
    rX, rZ = oracle.segment_summary(np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                                    np32(x["beta"]), cu)
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    assert rel_err(np32(X), rX) <= tol and rel_err(np32(Z), rZ) <= tol
    S_init = inputs.state(1, 2, 64, 64, seed=51, device=DEV)[0]
    E, Sf = B.scan_combine(X, Z, S_init)
    rE, rSf = oracle.scan_combine(np32(X), np32(Z), np32(S_init))
    assert rel_err(np32(E), rE) <= 1e-5 and rel_err(np32(Sf), rSf) <= 1e-5


def test_segment_summary_tensor_core_vs_oracle():
    """The tensor-core summary pass (bf16, d = 128): one CTA walks a chain's X and Z together.
    Ragged segments, an empty one (X = I, Z = 0 exactly) and a one-token one."""
    lengths = [100, 0, 64, 257, 1]
    x, cu = make_tokens(lengths, 3, 128, 128, torch.bfloat16, seed=52)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    X, Z = B.segment_summary(x["k"], x["v"], x["log_alpha"], x["beta"], cu_t)
    assert B.kda_get_error() == B.KDA_OK
    rX, rZ = oracle.segment_summary(np32(x["k"]), np32(x["v"]), np32(x["log_alpha"]),
                                    np32(x["beta"]), cu)
    check("summary_tc/X", np32(X), rX, TOL[torch.bfloat16])
    check("summary_tc/Z", np32(Z), rZ, TOL[torch.bfloat16])
    eye = torch.eye(128, device=DEV).expand(3, 128, 128)
    assert torch.equal(X[1], eye) and not Z[1].any()
    # the d = 128 scan over these summaries (tensor cores, split-bf16 products)
    S_init = inputs.state(1, 3, 128, 128, seed=53, device=DEV)[0]
    E, Sf = B.scan_combine(X, Z, S_init)
    rE, rSf = oracle.scan_combine(np32(X), np32(Z), np32(S_init))
    check("summary_tc/scan_E", np32(E), rE, 1e-5)
    check("summary_tc/scan_final", np32(Sf), rSf, 1e-5)


def _scan_inputs(n_seg, H, seed, d=128):
    """Contractive X (spectral norm about 0.9, as a segment's transition is) and Z, S_init of
    unit scale."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    X = torch.randn((n_seg, H, d, d), generator=g, device=DEV) / (2.2 * d ** 0.5)
    Z = torch.randn((n_seg, H, d, d), generator=g, device=DEV)
    S = torch.randn((H, d, d), generator=g, device=DEV)
    return X.contiguous(), Z.contiguous(), S


@pytest.mark.parametrize("n_seg", [0, 1, 2, 3, 8, 17])
@pytest.mark.parametrize("with_init", [False, True])
def test_scan_combine_d128_vs_oracle(n_seg, with_init):
    """kda_scan_combine at dk = dv = 128 (the tensor-core kernel: each fp32 operand as three
    bf16 terms, six products per step) against the oracle's fp64 scan at the fp32 tolerance.
    No segments, one segment (without S_init no product at all), and chains of 2 to 17 steps
    over 3 heads."""
    H = 3
    X, Z, S = _scan_inputs(n_seg, H, seed=60 + n_seg)
    S_init = S if with_init else None
    E, Sf = B.scan_combine(X, Z, S_init)
    assert B.kda_get_error() == B.KDA_OK
    rE, rSf = oracle.scan_combine(np32(X), np32(Z), None if S_init is None else np32(S_init))
    tag = f"scan_d128/n{n_seg}/{'init' if with_init else 'zero'}"
    if n_seg:
        check(tag + "/E", np32(E), rE, 1e-5)
    check(tag + "/final", np32(Sf), rSf, 1e-5)
    if not with_init and n_seg:
        assert not E[0].any()  # E_0 = 0 exactly
        if n_seg > 1:
            assert torch.equal(E[1], Z[0])  # E_1 = Z_0 exactly


def test_scan_combine_d128_one_output():
    """Entry states only, then the final state only: each equals the call that writes both."""
    n_seg, H = 5, 2
    X, Z, S = _scan_inputs(n_seg, H, seed=70)
    E, Sf = B.scan_combine(X, Z, S)
    E2 = torch.full_like(E, float("nan"))
    B.kda_scan_combine(X, Z, S, E2, None)
    Sf2 = torch.full_like(Sf, float("nan"))
    B.kda_scan_combine(X, Z, S, None, Sf2)
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(E2, E) and torch.equal(Sf2, Sf)


def test_context_parallel_driver_one_rank():
    """cp.context_parallel_forward with the device library on a one-rank NCCL group
    equals the monolithic chunked pass from the same initial state."""
    import socket

    import torch.distributed as dist

    from linear_attention_05_gb300 import cp
    with socket.socket() as sck:
        sck.bind(("127.0.0.1", 0))
        port = sck.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        x, _ = make_tokens([300], 4, 128, 128, torch.bfloat16, seed=60)
        S0 = inputs.state(1, 4, 128, 128, seed=61, device=DEV)
        out, s_mine, s_last = cp.context_parallel_forward(
            x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], S0[0].contiguous())
        ref_o, ref_s = gpu_chunk(x, [0, 300], S0=S0)
        assert rel_err(np32(out), np32(ref_o)) <= TOL[torch.bfloat16]
        assert rel_err(np32(s_mine), np32(ref_s[0])) <= TOL[torch.bfloat16]
        assert rel_err(np32(s_last), np32(ref_s[0])) <= TOL[torch.bfloat16]
    finally:
        dist.destroy_process_group()
