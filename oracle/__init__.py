"""KDA oracle: plain, slow, obviously-correct CPU reference (fp64).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The library path
never imports, links or calls it, and it imports nothing from the library.

Two independent restatements of the same definition live here:

* ``kda_oracle.c`` (loaded through ctypes): the token-by-token recurrence in
  its multiplied-out rank-1 form, S' = Diag(a) S; S = S' + b k (v - k^T S')^T;
  o = g * scale * S^T q, in double precision, OpenMP over (sequence, head).
* ``brute.py``: the same recurrence with the per-token transition built as an
  explicit dk x dk matrix, A_t = (I - b k k^T) Diag(a), in NumPy. Used on tiny
  cases to pin the C code.

``autograd.py`` holds the backward oracle: the recurrence once more in PyTorch
(fp64, CPU) and its gradients by torch.autograd, pinned to the C forward and to
finite differences of ``brute.py``. ``gates.py`` writes out the gate
preparation (sigmoid of the beta and output-gate logits, the lower-bounded
log-retention) used when the kernels take logits.

Definition sources: K3 training overview (zuoshipin.com/article/18261) section
2 "KDA" (channel-wise forget gate, delta-rule corrective write, full-rank
output gate) and section 3 "KDA context parallel" (per-segment transition and
zero-init state merged by an ordered prefix scan); K3 explainer
(devpress.csdn.net/awstech/6a72dc33...) section 2 (predict from memory, write
the error; delta rule with a channel-wise retention factor).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_default = None

L2_EPS = 1e-6  # eps inside the sqrt of the q/k L2 normalisation


def compile_source(src: str, out: str) -> str:
    """gcc -O2 (no fast-math) with OpenMP; returns the shared-object path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/ (skipped when up to date)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _f32(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


class Oracle:
    """ctypes view of one build of ``kda_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        i, d = ctypes.c_int, ctypes.c_double
        lib.kda_ref_forward.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i,
                                        d, i, P, P, P, i]
        lib.kda_ref_forward.restype = i
        lib.kda_ref_decode_step.argtypes = [P, P, P, P, P, P, P, P, i, i, i,
                                            i, d, i, P, i]
        lib.kda_ref_decode_step.restype = i
        lib.kda_ref_segment_summary.argtypes = [P, P, P, P, P, i, i, i, i,
                                                i, P, P, i]
        lib.kda_ref_segment_summary.restype = i
        lib.kda_ref_scan_combine.argtypes = [P, P, i, i, i, i, P, P, P]
        lib.kda_ref_scan_combine.restype = i
        lib.kda_ref_threads.argtypes = []
        lib.kda_ref_threads.restype = i
        self.lib = lib
        self.path = lib_path

    def threads(self) -> int:
        """Number of OpenMP threads the oracle uses by default."""
        return self.lib.kda_ref_threads()

    def forward(self, q, k, v, log_alpha, beta, gate=None, S0=None,
                cu_seqlens=None, scale=1.0, l2norm=True, t_stop=None,
                n_threads=0):
        """Full recurrence over packed sequences.

        q, k, log_alpha: [T_total, H, dk]; v, gate: [T_total, H, dv];
        beta: [T_total, H]; S0: [N_seq, H, dk, dv] or None (zero);
        cu_seqlens: [N_seq + 1] token offsets (None = one sequence);
        t_stop: optional per-sequence count of leading tokens to run.
        Returns (out [T_total, H, dv], S_final [N_seq, H, dk, dv]), fp64.
        """
        q, k, v, la, b, g = map(_f32, (q, k, v, log_alpha, beta, gate))
        T, H, dk = k.shape
        dv = v.shape[2]
        if cu_seqlens is None:
            cu_seqlens = [0, T]
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        n_seq = cu.shape[0] - 1
        S0 = _f64(S0)
        ts = None if t_stop is None else np.ascontiguousarray(
            np.asarray(t_stop, dtype=np.int64))
        out = np.zeros((T, H, dv), dtype=np.float64)
        Sf = np.zeros((n_seq, H, dk, dv), dtype=np.float64)
        rc = self.lib.kda_ref_forward(
            _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(g), _ptr(S0),
            _ptr(cu), n_seq, H, dk, dv, float(scale), int(bool(l2norm)),
            _ptr(out), _ptr(Sf), _ptr(ts), int(n_threads))
        if rc != 0:
            raise RuntimeError("kda_ref_forward failed")
        return out, Sf

    def decode_step(self, q, k, v, log_alpha, beta, gate, state, slot=None,
                    scale=1.0, l2norm=True, n_threads=0):
        """One token per sequence. ``state`` ([n_slots, H, dk, dv] fp64) is
        updated in place; returns out [N, H, dv] fp64."""
        q, k, v, la, b, g = map(_f32, (q, k, v, log_alpha, beta, gate))
        N, H, dk = k.shape
        dv = v.shape[2]
        if not (isinstance(state, np.ndarray) and state.dtype == np.float64
                and state.flags.c_contiguous):
            raise TypeError("state must be a C-contiguous float64 array")
        sl = None if slot is None else np.ascontiguousarray(
            np.asarray(slot, dtype=np.int64))
        out = np.zeros((N, H, dv), dtype=np.float64)
        rc = self.lib.kda_ref_decode_step(
            _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(g),
            _ptr(state), _ptr(sl), N, H, dk, dv, float(scale),
            int(bool(l2norm)), _ptr(out), int(n_threads))
        if rc != 0:
            raise RuntimeError("kda_ref_decode_step failed")
        return out

    def segment_summary(self, k, v, log_alpha, beta, cu_segs, l2norm=True,
                        n_threads=0):
        """Per-segment transition X [n_seg, H, dk, dk] and zero-init state
        Z [n_seg, H, dk, dv] (fp64), with S_out = X S_in + Z per head."""
        k, v, la, b = map(_f32, (k, v, log_alpha, beta))
        T, H, dk = k.shape
        dv = v.shape[2]
        cu = np.ascontiguousarray(np.asarray(cu_segs, dtype=np.int64))
        n_seg = cu.shape[0] - 1
        X = np.zeros((n_seg, H, dk, dk), dtype=np.float64)
        Z = np.zeros((n_seg, H, dk, dv), dtype=np.float64)
        rc = self.lib.kda_ref_segment_summary(
            _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(cu), n_seg, H, dk, dv,
            int(bool(l2norm)), _ptr(X), _ptr(Z), int(n_threads))
        if rc != 0:
            raise RuntimeError("kda_ref_segment_summary failed")
        return X, Z

    def scan_combine(self, X, Z, S_init=None):
        """Exclusive ordered scan: entry states E [n_seg, H, dk, dv] and the
        final state [H, dk, dv] (fp64)."""
        X, Z, S_init = _f64(X), _f64(Z), _f64(S_init)
        n_seg, H, dk, dv = Z.shape
        E = np.zeros_like(Z)
        Sf = np.zeros((H, dk, dv), dtype=np.float64)
        rc = self.lib.kda_ref_scan_combine(_ptr(X), _ptr(Z), n_seg, H, dk, dv,
                                           _ptr(S_init), _ptr(E), _ptr(Sf))
        if rc != 0:
            raise RuntimeError("kda_ref_scan_combine failed")
        return E, Sf


def default() -> Oracle:
    """The oracle built from ``kda_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def threads() -> int:
    return default().threads()


def forward(*a, **kw):
    return default().forward(*a, **kw)


def decode_step(*a, **kw):
    return default().decode_step(*a, **kw)


def segment_summary(*a, **kw):
    return default().segment_summary(*a, **kw)


def scan_combine(*a, **kw):
    return default().scan_combine(*a, **kw)
