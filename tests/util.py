"""Shared helpers for the tests (no KDA arithmetic here)."""
import numpy as np
import torch


def np32(t):
    """torch tensor (bf16 / fp32, any device) -> float32 NumPy array (exact for bf16)."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float32).numpy()


def rel_err(got, ref):
    """max |got - ref| / max |ref| over the whole tensor."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    if den == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / den)


# Tolerances (max|err| / max|ref| per output tensor): fp32 inputs 1e-4,
# bf16 inputs with fp32 state 2e-2.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def check(name, got, ref, tol):
    """Assert rel_err(got, ref) <= tol and print the margin as one greppable line
    ("PARITY <name> err=<e> tol=<t> margin=<tol/e>")."""
    e = rel_err(got, ref)
    margin = float("inf") if e == 0.0 else tol / e
    print(f"PARITY {name} err={e:.3e} tol={tol:.0e} margin={margin:.1f}x", flush=True)
    assert e <= tol, (name, e, tol)
    return e
