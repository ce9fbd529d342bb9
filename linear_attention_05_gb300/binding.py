"""ctypes binding over libkda: the C ABI's entry points under the same names.

Argument marshalling only. Every step of KDA runs in the library's CUDA
kernels; this module turns torch tensors into device pointers and sizes,
passes the current CUDA stream, and raises ``KdaError`` on a non-OK status.
There is no fallback: if ``libkda.so`` is missing or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libkda.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kda.h")

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3
KDA_ERR_TIMEOUT = 4
KDA_ERR_PRECONDITION = 5
KDA_ERR_WORKSPACE = 6
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED",
                3: "KDA_ERR_CUDA", 4: "KDA_ERR_TIMEOUT", 5: "KDA_ERR_PRECONDITION",
                6: "KDA_ERR_WORKSPACE"}
KDA_DTYPE_F32 = 0
KDA_DTYPE_BF16 = 1
KDA_QK_L2NORM = 1
KDA_DEBUG_CHECK = 2
KDA_GATE_LOGITS = 4
CHUNK = 64

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def declared_functions(header: str | None = None):
    """Names of the functions the headers in include/ declare (or one header)."""
    import glob
    paths = [header] if header else sorted(glob.glob(os.path.join(os.path.dirname(HEADER), "*.h")))
    names = set()
    for p in paths:
        txt = re.sub(r"/\*.*?\*/", "", open(p).read(), flags=re.S)
        names |= set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", txt))
    return sorted(names)


def load(path: str = LIB_PATH):
    """Load libkda.so (raises if it is missing) and declare the signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libkda.so not found at {path}; run linear_attention_05_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P, I, I64, F, U, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                               ctypes.c_uint, ctypes.c_size_t)
        sig = {
            "kda_version": ([], ctypes.c_char_p),
            "kda_last_error_string": ([], ctypes.c_char_p),
            "kda_chunk_fwd": ([P, P, P, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, U, I, P, SZ, P], I),
            "kda_chunk_fwd_workspace_size": ([I64, I, I, I, I, I, I], SZ),
            "kda_chunk_fwd_launches": ([I64, I, I, I, I, I, I, I], I),
            "kda_chunk_bwd": ([P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I64, I, I, I,
                               I, F, U, I, P, SZ, P], I),
            "kda_chunk_bwd_workspace_size": ([I64, I, I, I, I, I, I], SZ),
            "kda_segmented_fwd": ([P, P, P, P, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, U, I, P,
                                   SZ, P], I),
            "kda_segmented_fwd_workspace_size": ([I64, I, I, I, I, I, I], SZ),
            "kda_chunk_fwd_checkpoints": ([P, P, P, P, P, P, P, P, P, P, I64, I, P, I, I64, I, I,
                                           I, I, F, U, I, P, SZ, P], I),
            "kda_chunk_fwd_noalloc": ([P, P, P, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, U, I, P], I),
            "kda_chunk_fwd_host": ([P, P, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, U, I, I, P,
                                    SZ, P], I),
            "kda_chunk_fwd_host_buffer_size": ([I64, I, I, I, I, I, I, I], SZ),
            "kda_decode_step": ([P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, U, I, P], I),
            "kda_segment_summary": ([P, P, P, P, P, I, I64, I, I, I, I, U, I, P, P, P, SZ, P], I),
            "kda_segment_summary_workspace_size": ([I64, I, I, I, I, I, I], SZ),
            "kda_scan_combine": ([P, P, I, I, I, I, P, P, P, P], I),
            "kda_get_error": ([P], I),
            "kda_trace_events": ([ctypes.POINTER(P), ctypes.POINTER(P), I], I),
            "kda_selftest_umma": ([P, P, P, I, I, I, I, I, P], I),
            "kda_selftest_wait_timeout": ([U, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if t.numel() > 0 and not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_DTYPE_BF16
    if t.dtype == torch.float32:
        return KDA_DTYPE_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(lib, st: int):
    if st != KDA_OK:
        raise KdaError(st, lib.kda_last_error_string().decode())


def _f32_or_none(t, name):
    if t is not None and t.dtype != torch.float32:
        raise ValueError(f"{name} must be float32")
    return t


# ----------------------------------------------------------------------------- raw entry points
def kda_version() -> str:
    """Library version string."""
    return load().kda_version().decode()


def kda_last_error_string() -> str:
    return load().kda_last_error_string().decode()


def kda_chunk_fwd_workspace_size(T_total, n_seq, H, dk, dv, chunk=CHUNK, dtype=KDA_DTYPE_BF16):
    return int(load().kda_chunk_fwd_workspace_size(T_total, n_seq, H, dk, dv, chunk, dtype))


def kda_chunk_fwd_launches(T_total, n_seq, H, dk, dv, chunk=CHUNK, dtype=KDA_DTYPE_BF16,
                           varlen=False):
    """Kernel launches of kda_chunk_fwd for this problem (varlen: cu_seqlens given): 2 to 5,
    or 0 for an empty or invalid problem."""
    return int(load().kda_chunk_fwd_launches(T_total, n_seq, H, dk, dv, chunk, dtype,
                                             int(bool(varlen))))


def kda_segment_summary_workspace_size(T_total, n_seg, H, dk, dv, chunk=CHUNK, dtype=KDA_DTYPE_BF16):
    return int(load().kda_segment_summary_workspace_size(T_total, n_seg, H, dk, dv, chunk, dtype))


def _workspace(nbytes, device, workspace):
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    if nbytes == 0:
        return None, 0
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def kda_chunk_fwd(q, k, v, log_alpha, beta, gate, out, initial_state, final_state, cu_seqlens,
                  n_seq, scale=1.0, flags=KDA_QK_L2NORM, workspace=None, stream=None,
                  chunk=CHUNK):
    """Chunked prefill; writes ``out`` and (if given) ``final_state``."""
    lib = load()
    T, H, dk = k.shape
    dv = v.shape[-1]
    dt = _dtype_code(k)
    _f32_or_none(initial_state, "initial_state")
    _f32_or_none(final_state, "final_state")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    need = lib.kda_chunk_fwd_workspace_size(T, n_seq, H, dk, dv, chunk, dt)
    ws, wsb = _workspace(need, k.device, workspace)
    st = lib.kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(gate),
                           _ptr(out), _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens),
                           n_seq, T, H, dk, dv, chunk, float(scale), int(flags), dt, _ptr(ws),
                           wsb, _stream(stream))
    _check(lib, st)
    return out, final_state


def kda_chunk_fwd_checkpoints(q, k, v, log_alpha, beta, gate, out, initial_state, final_state,
                              checkpoints, checkpoint_every, cu_seqlens, n_seq, scale=1.0,
                              flags=KDA_QK_L2NORM, workspace=None, stream=None, chunk=CHUNK):
    """kda_chunk_fwd that also writes the state every ``checkpoint_every`` tokens into
    ``checkpoints`` [n_seq, per_seq, H, dk, dv] fp32 (or None for no checkpoints)."""
    lib = load()
    T, H, dk = k.shape
    dv = v.shape[-1]
    dt = _dtype_code(k)
    _f32_or_none(initial_state, "initial_state")
    _f32_or_none(final_state, "final_state")
    _f32_or_none(checkpoints, "checkpoints")
    per_seq = 0 if checkpoints is None else checkpoints.shape[1]
    if checkpoints is not None and tuple(checkpoints.shape) != (n_seq, per_seq, H, dk, dv):
        raise ValueError(f"checkpoints must be [n_seq, per_seq, H, dk, dv], got "
                         f"{tuple(checkpoints.shape)}")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    need = lib.kda_chunk_fwd_workspace_size(T, n_seq, H, dk, dv, chunk, dt)
    ws, wsb = _workspace(need, k.device, workspace)
    st = lib.kda_chunk_fwd_checkpoints(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(gate), _ptr(out),
        _ptr(initial_state), _ptr(final_state), _ptr(checkpoints), int(checkpoint_every),
        per_seq, _ptr(cu_seqlens), n_seq, T, H, dk, dv, chunk, float(scale), int(flags), dt,
        _ptr(ws), wsb, _stream(stream))
    _check(lib, st)
    return out, final_state, checkpoints


def kda_chunk_bwd_workspace_size(T_total, n_seq, H, dk, dv, chunk=CHUNK, dtype=KDA_DTYPE_BF16):
    return int(load().kda_chunk_bwd_workspace_size(T_total, n_seq, H, dk, dv, chunk, dtype))


def kda_chunk_bwd(q, k, v, log_alpha, beta, gate, initial_state, d_out, d_final_state, d_q, d_k,
                  d_v, d_log_alpha, d_beta, d_gate, d_initial_state, cu_seqlens, n_seq,
                  scale=1.0, flags=KDA_QK_L2NORM, workspace=None, stream=None, chunk=CHUNK):
    """Chunked backward pass; writes the gradient tensors passed in."""
    lib = load()
    T, H, dk = k.shape
    dv = v.shape[-1]
    dt = _dtype_code(k)
    for t, n in ((initial_state, "initial_state"), (d_final_state, "d_final_state"),
                 (d_initial_state, "d_initial_state")):
        _f32_or_none(t, n)
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    need = lib.kda_chunk_bwd_workspace_size(T, n_seq, H, dk, dv, chunk, dt)
    ws, wsb = _workspace(need, k.device, workspace)
    st = lib.kda_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(gate),
                           _ptr(initial_state), _ptr(d_out), _ptr(d_final_state), _ptr(d_q),
                           _ptr(d_k), _ptr(d_v), _ptr(d_log_alpha), _ptr(d_beta), _ptr(d_gate),
                           _ptr(d_initial_state), _ptr(cu_seqlens), n_seq, T, H, dk, dv, chunk,
                           float(scale), int(flags), dt, _ptr(ws), wsb, _stream(stream))
    _check(lib, st)


def kda_segmented_fwd_workspace_size(T_total, n_seg, H, dk, dv, chunk=CHUNK,
                                     dtype=KDA_DTYPE_BF16):
    return int(load().kda_segmented_fwd_workspace_size(T_total, n_seg, H, dk, dv, chunk, dtype))


def kda_segmented_fwd(q, k, v, log_alpha, beta, gate, out, initial_state, final_state,
                      segment_entry_states, cu_segs, n_seg, scale=1.0, flags=KDA_QK_L2NORM,
                      workspace=None, stream=None, chunk=CHUNK):
    """One sequence in n_seg segments: summaries, ordered scan, segment re-run (one card pass)."""
    lib = load()
    T, H, dk = k.shape
    dv = v.shape[-1]
    dt = _dtype_code(k)
    for t, n in ((initial_state, "initial_state"), (final_state, "final_state"),
                 (segment_entry_states, "segment_entry_states")):
        _f32_or_none(t, n)
    if cu_segs is not None and cu_segs.dtype != torch.int32:
        raise ValueError("cu_segs must be int32")
    need = lib.kda_segmented_fwd_workspace_size(T, n_seg, H, dk, dv, chunk, dt)
    ws, wsb = _workspace(need, k.device, workspace)
    st = lib.kda_segmented_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                               _ptr(gate), _ptr(out), _ptr(initial_state), _ptr(final_state),
                               _ptr(segment_entry_states), _ptr(cu_segs), n_seg, T, H, dk, dv,
                               chunk, float(scale), int(flags), dt, _ptr(ws), wsb,
                               _stream(stream))
    _check(lib, st)
    return out, final_state


def kda_chunk_fwd_noalloc(q, k, v, log_alpha, beta, gate, out, initial_state, final_state,
                          cu_seqlens, n_seq, scale=1.0, flags=KDA_QK_L2NORM, stream=None,
                          chunk=CHUNK):
    """kda_chunk_fwd using the library's fixed device scratch (no workspace).

    For callers that cannot allocate device memory where they run the mixer;
    the library allocates nothing either. Problems needing more than the fixed
    scratch raise KdaError(KDA_ERR_WORKSPACE). Calls that overlap on the GPU
    share the scratch and race."""
    lib = load()
    T, H, dk = k.shape
    dv = v.shape[-1]
    _f32_or_none(initial_state, "initial_state")
    _f32_or_none(final_state, "final_state")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    st = lib.kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                   _ptr(gate), _ptr(out), _ptr(initial_state), _ptr(final_state),
                                   _ptr(cu_seqlens), n_seq, T, H, dk, dv, chunk, float(scale),
                                   int(flags), _dtype_code(k), _stream(stream))
    _check(lib, st)
    return out, final_state


def _host_ptr(t):
    """Address of a contiguous CPU tensor (the library checks that it is page-locked)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if t.is_cuda:
        raise ValueError("tensor must be in host memory")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


def kda_chunk_fwd_host_buffer_size(T_total, n_seq, H, dk, dv, chunk=CHUNK,
                                   dtype=KDA_DTYPE_BF16, tail_slices=1):
    return int(load().kda_chunk_fwd_host_buffer_size(T_total, n_seq, H, dk, dv, chunk, dtype,
                                                     tail_slices))


def kda_chunk_fwd_host(q, k, v, log_alpha, beta, gate, out, initial_state, final_state, n_seq,
                       scale=1.0, flags=KDA_QK_L2NORM, tail_slices=1, device_buffer=None,
                       stream=None, chunk=CHUNK, device=None):
    """Prefill of ``n_seq`` equal-length sequences held in page-locked host tensors (e.g.
    ``torch.Tensor.pin_memory()``); writes the host tensors ``out`` and (if given)
    ``final_state``. The copies and the compute are queued on ``stream`` (and the library's
    copy streams); the host outputs are complete once ``stream`` has drained.
    ``device_buffer``: a CUDA uint8 tensor of at least kda_chunk_fwd_host_buffer_size bytes,
    allocated on ``device`` (default: the current device) when None."""
    lib = load()
    T, H, dk = k.shape
    dv = v.shape[-1]
    dt = _dtype_code(k)
    _f32_or_none(initial_state, "initial_state")
    _f32_or_none(final_state, "final_state")
    need = lib.kda_chunk_fwd_host_buffer_size(T, n_seq, H, dk, dv, chunk, dt, tail_slices)
    if device_buffer is None:
        dev = torch.device("cuda") if device is None else torch.device(device)
        device_buffer = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    nb = device_buffer.numel() * device_buffer.element_size()
    st = lib.kda_chunk_fwd_host(_host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(log_alpha),
                                _host_ptr(beta), _host_ptr(gate), _host_ptr(out),
                                _host_ptr(initial_state), _host_ptr(final_state), n_seq, T, H, dk,
                                dv, chunk, float(scale), int(flags), dt, int(tail_slices),
                                _ptr(device_buffer), nb, _stream(stream))
    _check(lib, st)
    return out, final_state


def kda_decode_step(q, k, v, log_alpha, beta, gate, out, state, state_slot=None, scale=1.0,
                    flags=KDA_QK_L2NORM, stream=None):
    """One token per sequence; updates ``state`` in place and writes ``out``."""
    lib = load()
    N, H, dk = k.shape
    dv = v.shape[-1]
    _f32_or_none(state, "state")
    if state_slot is not None and state_slot.dtype != torch.int32:
        raise ValueError("state_slot must be int32")
    st = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(gate),
                             _ptr(out), _ptr(state), _ptr(state_slot), state.shape[0], N, H, dk,
                             dv, float(scale), int(flags), _dtype_code(k), _stream(stream))
    _check(lib, st)
    return out


def kda_segment_summary(k, v, log_alpha, beta, cu_segs, n_seg, X_out, Z_out,
                        flags=KDA_QK_L2NORM, workspace=None, stream=None, chunk=CHUNK):
    """Per-segment transition X and zero-init state Z (fp32)."""
    lib = load()
    T, H, dk = k.shape
    dv = v.shape[-1]
    dt = _dtype_code(k)
    if cu_segs is not None and cu_segs.dtype != torch.int32:
        raise ValueError("cu_segs must be int32")
    need = lib.kda_segment_summary_workspace_size(T, n_seg, H, dk, dv, chunk, dt)
    ws, wsb = _workspace(need, k.device, workspace)
    st = lib.kda_segment_summary(_ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(cu_segs),
                                 n_seg, T, H, dk, dv, chunk, int(flags), dt, _ptr(X_out),
                                 _ptr(Z_out), _ptr(ws), wsb, _stream(stream))
    _check(lib, st)
    return X_out, Z_out


def kda_scan_combine(X, Z, S_init, S_entry_out, S_final_out, stream=None):
    """Ordered scan of the segment maps (fp32)."""
    lib = load()
    n_seg, H, dk, dv = Z.shape
    st = lib.kda_scan_combine(_ptr(X), _ptr(Z), n_seg, H, dk, dv, _ptr(S_init),
                              _ptr(S_entry_out), _ptr(S_final_out), _stream(stream))
    _check(lib, st)
    return S_entry_out, S_final_out


def kda_get_error(stream=None) -> int:
    """Synchronise the stream, read and clear the device error word; returns the status."""
    lib = load()
    return int(lib.kda_get_error(_stream(stream)))


def kda_trace_events(begin, end):
    """Record torch.cuda.Event pairs around each launch of later calls on this
    thread (begin[i]/end[i] around launch i); pass empty lists to stop."""
    lib = load()
    n = len(begin)
    if n != len(end):
        raise ValueError("begin and end must have the same length")
    for e in list(begin) + list(end):
        if e.cuda_event == 0:  # torch creates the event lazily
            e.record()
    arr_t = ctypes.c_void_p * max(n, 1)
    b = arr_t(*[e.cuda_event for e in begin])
    en = arr_t(*[e.cuda_event for e in end])
    _check(lib, lib.kda_trace_events(b, en, n))


def kda_selftest_umma(A, B, D, a_mn_major=0, b_mn_major=0, stream=None):
    """One tcgen05 product D = A @ B through the kernels' shared-memory tile
    layouts (diagnostic; see include/kda_selftest.h). Returns the status."""
    lib = load()
    M, K = A.shape
    N = B.shape[1]
    return int(lib.kda_selftest_umma(_ptr(A), _ptr(B), _ptr(D), M, N, K, int(a_mn_major),
                                     int(b_mn_major), _stream(stream)))


def kda_selftest_wait_timeout(limit_us, stream=None):
    """Launch the bounded-wait self-test (diagnostic; see include/kda_selftest.h): a wait that
    nothing completes runs out after ``limit_us`` and is reported by the next kda_get_error()."""
    lib = load()
    return int(lib.kda_selftest_wait_timeout(int(limit_us), _stream(stream)))


# ----------------------------------------------------------------------------- conveniences
def _flags(l2norm, gate_logits):
    return (KDA_QK_L2NORM if l2norm else 0) | (KDA_GATE_LOGITS if gate_logits else 0)


def chunk_fwd(q, k, v, log_alpha, beta, gate=None, initial_state=None, cu_seqlens=None,
              n_seq=None, scale=1.0, l2norm=True, output_final_state=True, workspace=None,
              stream=None, gate_logits=False):
    """Allocate the outputs with torch and call kda_chunk_fwd."""
    T, H, dk = k.shape
    dv = v.shape[-1]
    if n_seq is None:
        n_seq = (cu_seqlens.numel() - 1) if cu_seqlens is not None else 1
    out = torch.empty((T, H, dv), dtype=v.dtype, device=v.device)
    fs = (torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=v.device)
          if output_final_state else None)
    kda_chunk_fwd(q, k, v, log_alpha, beta, gate, out, initial_state, fs, cu_seqlens, n_seq,
                  scale=scale, flags=_flags(l2norm, gate_logits), workspace=workspace,
                  stream=stream)
    return out, fs


def chunk_fwd_checkpoints(q, k, v, log_alpha, beta, gate=None, initial_state=None,
                          cu_seqlens=None, n_seq=None, checkpoint_every=1024,
                          checkpoints_per_seq=None, scale=1.0, l2norm=True, workspace=None,
                          stream=None, gate_logits=False):
    """Allocate the outputs and call kda_chunk_fwd_checkpoints.

    Returns (out, final_state, checkpoints); checkpoints[s, i] is the state of sequence s
    after its first (i + 1) * checkpoint_every tokens. checkpoints_per_seq defaults to the
    longest sequence's count (reads cu_seqlens on the host)."""
    T, H, dk = k.shape
    dv = v.shape[-1]
    if n_seq is None:
        n_seq = (cu_seqlens.numel() - 1) if cu_seqlens is not None else 1
    if checkpoints_per_seq is None:
        if cu_seqlens is not None:
            longest = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if n_seq > 0 else 0
        else:
            longest = T // n_seq if n_seq > 0 else 0
        checkpoints_per_seq = longest // checkpoint_every
    out = torch.empty((T, H, dv), dtype=v.dtype, device=v.device)
    fs = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=v.device)
    ck = torch.zeros((n_seq, checkpoints_per_seq, H, dk, dv), dtype=torch.float32,
                     device=v.device)
    return kda_chunk_fwd_checkpoints(q, k, v, log_alpha, beta, gate, out, initial_state, fs,
                                     ck if checkpoints_per_seq > 0 else None, checkpoint_every,
                                     cu_seqlens, n_seq, scale=scale,
                                     flags=_flags(l2norm, gate_logits), workspace=workspace,
                                     stream=stream)[:2] + (ck,)


def chunk_bwd(q, k, v, log_alpha, beta, gate, initial_state, d_out, d_final_state=None,
              cu_seqlens=None, n_seq=None, scale=1.0, l2norm=True, workspace=None, stream=None,
              gate_logits=False):
    """Allocate the gradients and call kda_chunk_bwd. Returns a dict with dq, dk, dv,
    dlog_alpha, dbeta, dgate (None without a gate) and dS0 (fp32)."""
    T, H, dk = k.shape
    dv = v.shape[-1]
    if n_seq is None:
        n_seq = (cu_seqlens.numel() - 1) if cu_seqlens is not None else 1
    g = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
         "dlog_alpha": torch.empty_like(log_alpha), "dbeta": torch.empty_like(beta),
         "dgate": None if gate is None else torch.empty_like(gate),
         "dS0": torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=k.device)}
    kda_chunk_bwd(q, k, v, log_alpha, beta, gate, initial_state, d_out, d_final_state, g["dq"],
                  g["dk"], g["dv"], g["dlog_alpha"], g["dbeta"], g["dgate"], g["dS0"],
                  cu_seqlens, n_seq, scale=scale, flags=_flags(l2norm, gate_logits),
                  workspace=workspace, stream=stream)
    return g


def segmented_fwd(q, k, v, log_alpha, beta, gate=None, initial_state=None, cu_segs=None,
                  n_seg=None, scale=1.0, l2norm=True, gate_logits=False, workspace=None,
                  stream=None):
    """Allocate out, the final state and the segment entry states; call kda_segmented_fwd.
    Returns (out, final_state [H, dk, dv], entry_states [n_seg, H, dk, dv])."""
    T, H, dk = k.shape
    dv = v.shape[-1]
    if n_seg is None:
        n_seg = cu_segs.numel() - 1
    out = torch.empty((T, H, dv), dtype=v.dtype, device=v.device)
    fs = torch.empty((H, dk, dv), dtype=torch.float32, device=v.device)
    ent = torch.empty((n_seg, H, dk, dv), dtype=torch.float32, device=v.device)
    kda_segmented_fwd(q, k, v, log_alpha, beta, gate, out, initial_state, fs, ent, cu_segs, n_seg,
                      scale=scale, flags=_flags(l2norm, gate_logits), workspace=workspace,
                      stream=stream)
    return out, fs, ent


def decode_step(q, k, v, log_alpha, beta, gate, state, state_slot=None, scale=1.0, l2norm=True,
                stream=None, gate_logits=False):
    out = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    return kda_decode_step(q, k, v, log_alpha, beta, gate, out, state, state_slot, scale,
                           _flags(l2norm, gate_logits), stream)


def segment_summary(k, v, log_alpha, beta, cu_segs, l2norm=True, workspace=None, stream=None,
                    gate_logits=False):
    n_seg = cu_segs.numel() - 1
    T, H, dk = k.shape
    dv = v.shape[-1]
    X = torch.empty((n_seg, H, dk, dk), dtype=torch.float32, device=k.device)
    Z = torch.empty((n_seg, H, dk, dv), dtype=torch.float32, device=k.device)
    return kda_segment_summary(k, v, log_alpha, beta, cu_segs, n_seg, X, Z,
                               _flags(l2norm, gate_logits), workspace, stream)


def scan_combine(X, Z, S_init=None, stream=None):
    n_seg, H, dk, dv = Z.shape
    E = torch.empty_like(Z)
    Sf = torch.empty((H, dk, dv), dtype=torch.float32, device=Z.device)
    return kda_scan_combine(X, Z, S_init, E, Sf, stream)
