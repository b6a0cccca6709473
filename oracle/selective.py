"""Float64 oracle for the Mamba-1 selective scan -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference legs may
import this module.  It shares no code with the CUDA path.

Source: "3.3 Hardware-aware algorithm and GPU memory hierarchy" (booiljung.github.io),
section 2.1 (zero-order-hold discretisation Abar = exp(delta A), Bbar = (delta A)^-1
(exp(delta A) - I) delta B; only y leaves the fused kernel), section 3 (load,
discretise, scan, multiply by C) and section 4.1 (h_t = Abar_t h_{t-1} + Bbar_t x_t).

Conventions: x, delta, y (b, L, D); B, C (b, L, N); A (D, N); Dskip (D); init / final
(b, D, N).  x, delta, B, C are float32 or bfloat16 bit patterns (uint16), widened exactly.
"""
import ctypes

import numpy as np

from . import ref as _ref

_BOUND = False


def _lib():
    global _BOUND
    lib = _ref._lib()
    if not _BOUND:
        vp = ctypes.c_void_p
        lib.ssd_ref_selective_scan.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int] + [vp] * 9
        lib.ssd_ref_selective_scan.restype = ctypes.c_int
        _BOUND = True
    return lib


def _io(a, want):
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError("x, delta, B, C must share one dtype (float32 or bf16 bits as uint16)")
    return a


def selective_scan(x, delta, A, B, C, Dskip=None, init=None, want_final=True):
    """Token-by-token selective scan in float64 (C, OpenMP over channels).

    Returns dict(y (b, L, D) float64, final (b, D, N) float64 if want_final).
    """
    bf16 = np.asarray(x).dtype == np.uint16
    want = np.uint16 if bf16 else np.float32
    x, delta, B, C = (_io(a, want) for a in (x, delta, B, C))
    b, L, D = x.shape
    N = B.shape[2]
    if delta.shape != x.shape or B.shape != (b, L, N) or C.shape != (b, L, N):
        raise ValueError("shape mismatch")
    A = np.ascontiguousarray(A, np.float32)
    Dskip = None if Dskip is None else np.ascontiguousarray(Dskip, np.float32)
    init = None if init is None else np.ascontiguousarray(init, np.float32)
    y = np.empty((b, L, D))
    fin = np.empty((b, D, N)) if want_final else None
    p = _ref._ptr
    rc = _lib().ssd_ref_selective_scan(b, L, D, N, int(bf16), p(x), p(delta), p(A), p(B), p(C),
                                       p(Dskip), p(init), p(y), p(fin))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    out = {"y": y}
    if want_final:
        out["final"] = fin
    return out


def selective_scan_np(x, delta, A, B, C, Dskip=None, init=None):
    """NumPy twin of the C oracle for small inputs: (y (b, L, D), final (b, D, N)).

    Same definition, vectorised over (b, d, n), looping over tokens.
    """
    x, delta, B, C = (_ref.widen(a) for a in (x, delta, B, C))
    A = np.asarray(A, np.float64)
    b, L, D = x.shape
    N = B.shape[2]
    h = np.zeros((b, D, N)) if init is None else np.asarray(init, np.float64).copy()
    skip = np.zeros(D) if Dskip is None else np.asarray(Dskip, np.float64)
    y = np.empty((b, L, D))
    for t in range(L):
        w = delta[:, t, :, None] * A[None]                           # (b, D, N)
        safe = np.where(A == 0.0, 1.0, A)
        coef = np.where(A[None] == 0.0, delta[:, t, :, None], np.expm1(w) / safe[None])
        h = np.exp(w) * h + coef * B[:, t, None, :] * x[:, t, :, None]
        y[:, t] = np.einsum("bdn,bn->bd", h, C[:, t]) + skip * x[:, t]
    return y, h
