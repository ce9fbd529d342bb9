"""The C ABI without a GPU: the library loads, exports what include/kda.h
declares, and rejects bad arguments with the documented status before any
CUDA call."""
import ctypes

import pytest

from linear_attention_05_gb300 import binding as B


@pytest.fixture(scope="module")
def lib():
    return B.load()


def test_exports_every_declared_symbol(lib):
    names = B.declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert "sm_103a" in B.kda_version()


FAKE = 0x10000  # never dereferenced: every call below fails validation first
ODD = 0x10001


def chunk(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, la=FAKE, beta=FAKE, gate=None, out=FAKE, s0=None, sf=None,
             cu=None, n_seq=1, T=128, H=2, dk=64, dv=64, chunk=64, scale=1.0, flags=1,
             dtype=1, ws=FAKE, wsb=0, stream=None)
    a.update(kw)
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["la"], a["beta"], a["gate"], a["out"],
                             a["s0"], a["sf"], a["cu"], a["n_seq"], a["T"], a["H"], a["dk"],
                             a["dv"], a["chunk"], a["scale"], a["flags"], a["dtype"], a["ws"],
                             a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dk=96), B.KDA_ERR_UNSUPPORTED),
    (dict(dv=256), B.KDA_ERR_UNSUPPORTED),
    (dict(chunk=32), B.KDA_ERR_UNSUPPORTED),
    (dict(dtype=7), B.KDA_ERR_UNSUPPORTED),
    (dict(T=-1), B.KDA_ERR_INVALID_ARG),
    (dict(H=0), B.KDA_ERR_INVALID_ARG),
    (dict(n_seq=-2), B.KDA_ERR_INVALID_ARG),
    (dict(q=None), B.KDA_ERR_INVALID_ARG),
    (dict(beta=None), B.KDA_ERR_INVALID_ARG),
    (dict(out=None), B.KDA_ERR_INVALID_ARG),
    (dict(k=ODD), B.KDA_ERR_INVALID_ARG),
    (dict(gate=ODD), B.KDA_ERR_INVALID_ARG),
    (dict(sf=ODD), B.KDA_ERR_INVALID_ARG),
    (dict(cu=FAKE + 2), B.KDA_ERR_INVALID_ARG),
    (dict(n_seq=3, T=128), B.KDA_ERR_INVALID_ARG),  # 128 tokens do not split into 3 equal seqs
    (dict(flags=0x80), B.KDA_ERR_INVALID_ARG),
    (dict(ws=None, wsb=0), B.KDA_ERR_WORKSPACE),
    (dict(wsb=100), B.KDA_ERR_WORKSPACE),
])
def test_chunk_fwd_rejects(lib, kw, status):
    assert chunk(lib, **kw) == status
    assert B.kda_last_error_string() != ""


def test_chunk_fwd_no_sequences_is_noop(lib):
    assert chunk(lib, n_seq=0, T=0, q=None, k=None, v=None, la=None, beta=None, out=None,
                 ws=None) == B.KDA_OK


def ckpt(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, la=FAKE, beta=FAKE, gate=None, out=FAKE, s0=None, sf=None,
             cp=FAKE, every=128, per=2, cu=None, n_seq=1, T=256, H=2, dk=64, dv=64, chunk=64,
             scale=1.0, flags=1, dtype=1, ws=FAKE, wsb=0, stream=None)
    a.update(kw)
    return lib.kda_chunk_fwd_checkpoints(
        a["q"], a["k"], a["v"], a["la"], a["beta"], a["gate"], a["out"], a["s0"], a["sf"],
        a["cp"], a["every"], a["per"], a["cu"], a["n_seq"], a["T"], a["H"], a["dk"], a["dv"],
        a["chunk"], a["scale"], a["flags"], a["dtype"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(every=0), B.KDA_ERR_INVALID_ARG),
    (dict(every=-64), B.KDA_ERR_INVALID_ARG),
    (dict(every=100), B.KDA_ERR_INVALID_ARG),     # not a multiple of the chunk
    (dict(every=64 * (2 ** 31)), B.KDA_ERR_INVALID_ARG),  # spacing in chunks overflows int
    (dict(per=-1), B.KDA_ERR_INVALID_ARG),
    (dict(cp=None), B.KDA_ERR_INVALID_ARG),       # slots requested, no buffer
    (dict(cp=ODD), B.KDA_ERR_INVALID_ARG),
    (dict(dk=96), B.KDA_ERR_UNSUPPORTED),         # then every kda_chunk_fwd check
    (dict(ws=None), B.KDA_ERR_WORKSPACE),
])
def test_chunk_fwd_checkpoints_rejects(lib, kw, status):
    assert ckpt(lib, **kw) == status
    assert B.kda_last_error_string() != ""


def test_chunk_fwd_checkpoints_no_sequences_is_noop(lib):
    # zero slots: the buffer may be NULL; no sequences: nothing runs
    assert ckpt(lib, cp=None, per=0, n_seq=0, T=0, q=None, k=None, v=None, la=None, beta=None,
                out=None, ws=None) == B.KDA_OK


def bwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, la=FAKE, beta=FAKE, gate=FAKE, s0=None, dout=FAKE,
             dsf=None, dq=FAKE, dk_=FAKE, dv_=FAKE, dla=FAKE, db=FAKE, dg=FAKE, ds0=None,
             cu=None, n_seq=1, T=128, H=2, dk=64, dv=64, chunk=64, scale=1.0, flags=1, dtype=1,
             ws=FAKE, wsb=0, stream=None)
    a.update(kw)
    return lib.kda_chunk_bwd(a["q"], a["k"], a["v"], a["la"], a["beta"], a["gate"], a["s0"],
                             a["dout"], a["dsf"], a["dq"], a["dk_"], a["dv_"], a["dla"], a["db"],
                             a["dg"], a["ds0"], a["cu"], a["n_seq"], a["T"], a["H"], a["dk"],
                             a["dv"], a["chunk"], a["scale"], a["flags"], a["dtype"], a["ws"],
                             a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dk=32), B.KDA_ERR_UNSUPPORTED),
    (dict(chunk=128), B.KDA_ERR_UNSUPPORTED),
    (dict(T=-5), B.KDA_ERR_INVALID_ARG),
    (dict(dout=None), B.KDA_ERR_INVALID_ARG),
    (dict(dq=None), B.KDA_ERR_INVALID_ARG),
    (dict(db=None), B.KDA_ERR_INVALID_ARG),
    (dict(dla=ODD), B.KDA_ERR_INVALID_ARG),
    (dict(gate=None), B.KDA_ERR_INVALID_ARG),   # d_gate without a gate
    (dict(dsf=ODD), B.KDA_ERR_INVALID_ARG),
    (dict(flags=8), B.KDA_ERR_INVALID_ARG),
    (dict(ws=None), B.KDA_ERR_WORKSPACE),
    (dict(wsb=1000), B.KDA_ERR_WORKSPACE),
])
def test_chunk_bwd_rejects(lib, kw, status):
    assert bwd(lib, **kw) == status
    assert B.kda_last_error_string() != ""


def test_chunk_bwd_workspace_size(lib):
    fw = B.kda_chunk_fwd_workspace_size(4096, 1, 16, 128, 128, dtype=B.KDA_DTYPE_F32)
    bw = B.kda_chunk_bwd_workspace_size(4096, 1, 16, 128, 128)
    assert bw > fw > 0
    assert B.kda_chunk_bwd_workspace_size(4096, 1, 16, 96, 128) == 0


def test_segmented_fwd_rejects(lib):
    args = lambda **kw: [kw.get(n, d) for n, d in (
        ("q", FAKE), ("k", FAKE), ("v", FAKE), ("la", FAKE), ("beta", FAKE), ("gate", None),
        ("out", FAKE), ("s0", None), ("sf", None), ("ent", None), ("cu", None), ("n_seg", 2),
        ("T", 256), ("H", 2), ("dk", 64), ("dv", 64), ("chunk", 64), ("scale", 1.0),
        ("flags", 1), ("dtype", 1), ("ws", FAKE), ("wsb", 0), ("stream", None))]
    assert lib.kda_segmented_fwd(*args(n_seg=0, T=0)) == B.KDA_ERR_INVALID_ARG
    assert lib.kda_segmented_fwd(*args(ent=ODD)) == B.KDA_ERR_INVALID_ARG
    assert lib.kda_segmented_fwd(*args(dv=32)) == B.KDA_ERR_UNSUPPORTED
    assert lib.kda_segmented_fwd(*args()) == B.KDA_ERR_WORKSPACE
    assert (B.kda_segmented_fwd_workspace_size(256, 2, 2, 64, 64)
            > B.kda_chunk_fwd_workspace_size(256, 2, 2, 64, 64))


def test_workspace_size(lib):
    s1 = B.kda_chunk_fwd_workspace_size(4096, 1, 16, 128, 128)
    s2 = B.kda_chunk_fwd_workspace_size(8192, 1, 16, 128, 128)
    assert 0 < s1 < s2
    assert B.kda_chunk_fwd_workspace_size(4096, 1, 16, 96, 128) == 0
    assert B.kda_segment_summary_workspace_size(4096, 2, 16, 128, 128) > 0


def test_chunk_fwd_launches(lib):
    """Prefills with few (sequence, head) pairs and long sequences are split (two card and two
    state launches instead of one each); the tensor-core path (bf16, d = 128) skips the chunk
    table without cu_seqlens; every other shape or dtype takes table, prep and state pass."""
    bf, f32 = B.KDA_DTYPE_BF16, B.KDA_DTYPE_F32
    L = B.kda_chunk_fwd_launches
    assert L(4 * 4096, 4, 16, 128, 128, dtype=bf) == 4
    assert L(4 * 4096, 4, 16, 128, 128, dtype=bf, varlen=True) == 5
    assert L(16 * 1024, 7, 16, 128, 128, dtype=bf, varlen=True) == 5     # 112 pairs
    assert L(16 * 1024, 8, 16, 128, 128, dtype=bf, varlen=True) == 3     # 128 pairs
    assert L(16 * 1024, 8, 16, 128, 128, dtype=bf) == 2
    assert L(4 * 512, 4, 16, 128, 128, dtype=bf, varlen=True) == 3       # 8 chunks/seq
    assert L(4 * 1024, 4, 16, 128, 128, dtype=bf) == 4                   # 16 chunks/seq
    assert L(4 * 4096, 4, 16, 128, 128, dtype=f32) == 3
    assert L(4 * 4096, 4, 16, 128, 128, dtype=f32, varlen=True) == 3
    assert L(4 * 4096, 4, 16, 64, 64, dtype=bf) == 3
    assert B.kda_chunk_fwd_launches(0, 0, 16, 128, 128, dtype=bf) == 0
    assert B.kda_chunk_fwd_launches(4096, 1, 16, 96, 128, dtype=bf) == 0
    # a split prefill's workspace holds the hand-over state between the parts
    split = B.kda_chunk_fwd_workspace_size(4 * 1024, 4, 16, 128, 128)
    whole = B.kda_chunk_fwd_workspace_size(4 * 1024 - 64, 4, 16, 128, 128)
    assert split - whole >= 4 * 16 * 128 * 128 * 4


def dec(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, la=FAKE, beta=FAKE, gate=None, out=FAKE, state=FAKE,
             slot=None, n_slots=4, N=4, H=2, dk=128, dv=128, scale=1.0, flags=1, dtype=1,
             stream=None)
    a.update(kw)
    return lib.kda_decode_step(a["q"], a["k"], a["v"], a["la"], a["beta"], a["gate"], a["out"],
                               a["state"], a["slot"], a["n_slots"], a["N"], a["H"], a["dk"],
                               a["dv"], a["scale"], a["flags"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dk=32), B.KDA_ERR_UNSUPPORTED),
    (dict(N=-1), B.KDA_ERR_INVALID_ARG),
    (dict(state=None), B.KDA_ERR_INVALID_ARG),
    (dict(state=ODD), B.KDA_ERR_INVALID_ARG),
    (dict(n_slots=2), B.KDA_ERR_INVALID_ARG),  # fewer slots than sequences, no slot map
    (dict(slot=FAKE + 1), B.KDA_ERR_INVALID_ARG),
    (dict(flags=8), B.KDA_ERR_INVALID_ARG),
])
def test_decode_rejects(lib, kw, status):
    assert dec(lib, **kw) == status


def test_decode_zero_sequences_is_noop(lib):
    assert dec(lib, N=0, q=None) == B.KDA_OK


def test_segment_summary_rejects(lib):
    st = lib.kda_segment_summary(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 256, 2, 64, 64, 64, 1, 1,
                                 FAKE, FAKE, FAKE, 10, None)
    assert st == B.KDA_ERR_WORKSPACE
    st = lib.kda_segment_summary(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 256, 2, 64, 64, 48, 1, 1,
                                 FAKE, FAKE, FAKE, 10, None)
    assert st == B.KDA_ERR_UNSUPPORTED


def test_scan_combine_rejects(lib):
    assert lib.kda_scan_combine(None, FAKE, 2, 2, 64, 64, None, FAKE, None, None) == \
        B.KDA_ERR_INVALID_ARG
    assert lib.kda_scan_combine(FAKE, FAKE, 2, 2, 64, 80, None, FAKE, None, None) == \
        B.KDA_ERR_UNSUPPORTED
    # nothing requested: a no-op
    assert lib.kda_scan_combine(FAKE, FAKE, 2, 2, 64, 64, None, None, None, None) == B.KDA_OK


def test_selftest_wait_timeout_rejects_bad_limit(lib):
    # checked before any launch: no GPU needed
    assert lib.kda_selftest_wait_timeout(0, None) == B.KDA_ERR_INVALID_ARG
    assert lib.kda_selftest_wait_timeout(2_000_000, None) == B.KDA_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    """No fallback: with libkda.so absent, loading raises (in a fresh process, so that this
    session's loaded handle is not reused)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys\n"
            "from linear_attention_05_gb300 import binding as B\n"
            "try:\n"
            f"    B.load({str(tmp_path / 'libkda.so')!r})\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n"
            "    sys.exit(0)\n"
            "sys.exit(1)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "not found" in r.stdout


def host_fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, la=FAKE, beta=FAKE, gate=None, out=FAKE, s0=None, sf=None,
             n_seq=2, T=256, H=2, dk=64, dv=64, chunk=64, scale=1.0, flags=1, dtype=1, tail=1,
             buf=None, bufb=0, stream=None)
    a.update(kw)
    return lib.kda_chunk_fwd_host(a["q"], a["k"], a["v"], a["la"], a["beta"], a["gate"],
                                  a["out"], a["s0"], a["sf"], a["n_seq"], a["T"], a["H"], a["dk"],
                                  a["dv"], a["chunk"], a["scale"], a["flags"], a["dtype"],
                                  a["tail"], a["buf"], a["bufb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dk=96), B.KDA_ERR_UNSUPPORTED),
    (dict(chunk=32), B.KDA_ERR_UNSUPPORTED),
    (dict(n_seq=0), B.KDA_ERR_INVALID_ARG),
    (dict(n_seq=3), B.KDA_ERR_INVALID_ARG),           # 256 tokens do not split into 3
    (dict(tail=0), B.KDA_ERR_INVALID_ARG),
    (dict(tail=17), B.KDA_ERR_INVALID_ARG),
    (dict(tail=4), B.KDA_ERR_INVALID_ARG),            # 128 tokens a sequence: not 4 x 64
    (dict(buf=None, bufb=0), B.KDA_ERR_WORKSPACE),
    (dict(buf=FAKE, bufb=100), B.KDA_ERR_WORKSPACE),
    (dict(buf=FAKE + 16, bufb=1 << 40), B.KDA_ERR_INVALID_ARG),   # not 256-byte aligned
    (dict(q=None, buf=FAKE, bufb=1 << 40), B.KDA_ERR_INVALID_ARG),
    (dict(out=None, buf=FAKE, bufb=1 << 40), B.KDA_ERR_INVALID_ARG),
])
def test_chunk_fwd_host_rejects(lib, kw, status):
    """kda_chunk_fwd_host's argument errors, all found before any CUDA call."""
    assert host_fwd(lib, **kw) == status
    assert b"kda_chunk_fwd_host" in lib.kda_last_error_string()


def test_chunk_fwd_host_buffer_size(lib):
    """The device buffer holds a slot per sequence for every tensor (256-byte aligned), the
    states and one sequence's workspace; invalid problems give 0."""
    S = B.kda_chunk_fwd_host_buffer_size
    n, L, H, d = 4, 4096, 16, 128
    size = S(n * L, n, H, d, d, tail_slices=4)
    staging = n * L * H * (5 * d + 1 + d) * 2 + 2 * n * H * d * d * 4
    ws = B.kda_chunk_fwd_workspace_size(L, 1, H, d, d)   # one sequence's update cards
    assert staging + ws <= size < staging + ws + (4 << 20)  # + the two hand-over states
    assert S(n * L, n, H, d, d, tail_slices=1) > 0
    assert S(3 * 77, 3, 5, 64, 64, tail_slices=1) > 0      # any length with one slice
    assert S(3 * 77, 3, 5, 64, 64, tail_slices=2) == 0     # slices need 64-token multiples
    assert S(n * L, n, H, 96, d) == 0
    assert S(n * L + 1, n, H, d, d) == 0
    assert S(n * L, n, H, d, d, tail_slices=32) == 0
