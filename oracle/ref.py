"""Float64 oracle for the Mamba-2 SSD forward scan -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
legs may import this module.  It shares no code with the CUDA path.

Sources (web pages this project follows):
  [P1] "Mamba-2 cuda-tile forward pass kernels" (devotd.net): section 1 (the
       recurrence is turned into per-chunk matrix products), section 2 (the
       chunk_cumsum kernel and its listing: an in-chunk cumulative sum of A*dt
       over the chunk axis, scaled by log2(e), zero-padded past the sequence;
       fwd_pass_state: the state entering each chunk and the state after the
       last one; compute_out: outputs from the chunk-start states).
  [P3] "Compiler-First State Space Duality and Portable O(1) Autoregressive
       Caching" (gist.science summary), technical summary section 2: chunking,
       batched einsums, static causal masks, decay kept in wide precision.

Conventions: x (b,L,H,P), dt (b,L,H), A (H), B and C (b,L,G,N), D (H),
init / final state (b,H,P,N); head h reads group g = h // (H // G).  x, B, C
are float32 arrays or bfloat16 bit patterns (uint16); everything is widened
exactly to float64 before any arithmetic.
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

LOG2E = 1.4426950408889634  # log2(e): [P1] section 2 scales the cumsum by it


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups", "chunk")]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(_build.build())
        vp, fp, dp, ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        lib.ssd_ref_recurrence.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int, vp, fp, fp, vp, vp,
                                           fp, fp, ip, ctypes.c_int64, dp, dp, dp]
        lib.ssd_ref_recurrence.restype = ctypes.c_int
        lib.ssd_ref_chunk_states.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int, vp, fp, fp, vp,
                                             ip, ctypes.c_int64, dp]
        lib.ssd_ref_chunk_states.restype = ctypes.c_int
        lib.ssd_ref_num_threads.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def num_threads() -> int:
    """OpenMP threads the C oracle runs on."""
    return int(_lib().ssd_ref_num_threads())


def widen(a) -> np.ndarray:
    """float32 array or bfloat16 bit pattern (uint16) -> float64, exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _io_arrays(x, B, C):
    bf16 = np.asarray(x).dtype == np.uint16
    want = np.uint16 if bf16 else np.float32
    out = []
    for a in (x, B, C):
        a = np.ascontiguousarray(a)
        if a.dtype != want:
            raise TypeError("x, B, C must share one dtype (float32 or bf16 bits as uint16)")
        out.append(a)
    return bf16, out


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _dims(x, B, chunk):
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return _Dims(b, L, H, P, N, G, chunk)


def all_pairs(batch, nheads):
    return np.array([(b, h) for b in range(batch) for h in range(nheads)], dtype=np.int64)


def recurrence(x, dt, A, B, C, D=None, init=None, chunk=256, pairs=None, want_y=True,
               want_final=True, want_chunk_in=False):
    """Token-by-token recurrence in float64 (C, OpenMP) for the selected (b, h) pairs.

    Follows [P1] sections 1-2: h_t = exp(dt_t A_h) h_{t-1} + dt_t x_t (x) B_t and
    y_t = C_t . h_t + D_h x_t.  Returns dict with
      y        (nsel, L, P)       if want_y
      final    (nsel, P, N)       if want_final  (state after the last token)
      chunk_in (nsel, nc, P, N)   if want_chunk_in (state entering chunk c)
    pairs defaults to every (b, h) in row-major order.
    """
    bf16, (x, B, C) = _io_arrays(x, B, C)
    dt, A, D, init = _f32(dt), _f32(A), _f32(D), _f32(init)
    d = _dims(x, B, chunk)
    pairs = all_pairs(d.batch, d.nheads) if pairs is None else np.ascontiguousarray(pairs, np.int64)
    nsel = pairs.shape[0]
    nc = (d.seqlen + chunk - 1) // chunk
    y = np.empty((nsel, d.seqlen, d.headdim)) if want_y else None
    fin = np.empty((nsel, d.headdim, d.dstate)) if want_final else None
    cin = np.empty((nsel, nc, d.headdim, d.dstate)) if want_chunk_in else None
    rc = _lib().ssd_ref_recurrence(ctypes.byref(d), int(bf16), _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                   _ptr(C), _ptr(D), _ptr(init), _ptr(pairs), nsel, _ptr(y),
                                   _ptr(fin), _ptr(cin))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    out = {}
    if want_y:
        out["y"] = y
    if want_final:
        out["final"] = fin
    if want_chunk_in:
        out["chunk_in"] = cin
    return out


def chunk_states(x, dt, A, B, chunk, pairs=None):
    """Per-chunk end state started from zero, (nsel, nc, P, N), float64.

    The quantity [P1] section 2's second kernel accumulates per chunk before
    chaining: the recurrence run over one chunk's tokens from h = 0.
    """
    bf16, (x, B, _) = _io_arrays(x, B, B)
    dt, A = _f32(dt), _f32(A)
    d = _dims(x, B, chunk)
    pairs = all_pairs(d.batch, d.nheads) if pairs is None else np.ascontiguousarray(pairs, np.int64)
    nc = (d.seqlen + chunk - 1) // chunk
    S = np.empty((pairs.shape[0], nc, d.headdim, d.dstate))
    rc = _lib().ssd_ref_chunk_states(ctypes.byref(d), int(bf16), _ptr(x), _ptr(dt), _ptr(A),
                                     _ptr(B), _ptr(pairs), pairs.shape[0], _ptr(S))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return S


def recurrence_np(x, dt, A, B, C, D=None, init=None):
    """NumPy twin of the C recurrence for tiny inputs: (y (b,L,H,P), final (b,H,P,N)).

    Same definition as ``recurrence`` ([P1] sections 1-2), vectorised over
    (b, h, p, n) and looping over tokens.
    """
    x, B, C = widen(x), widen(B), widen(C)
    dt, A = np.asarray(dt, np.float64), np.asarray(A, np.float64)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    grp = np.arange(H) // (H // G)
    Dv = np.zeros(H) if D is None else np.asarray(D, np.float64)
    h = np.zeros((b, H, P, N)) if init is None else np.asarray(init, np.float64).copy()
    y = np.empty((b, L, H, P))
    for t in range(L):
        Bt, Ct = B[:, t][:, grp], C[:, t][:, grp]          # (b, H, N)
        decay = np.exp(dt[:, t] * A)                        # (b, H)
        h = decay[..., None, None] * h + (dt[:, t][..., None] * x[:, t])[..., None] * Bt[:, :, None, :]
        y[:, t] = np.einsum("bhpn,bhn->bhp", h, Ct) + Dv[:, None] * x[:, t]
    return y, h


def cumsum_log2(dt, A, chunk):
    """In-chunk inclusive cumsum of A*dt in the log2 domain, float64.

    [P1] section 2 and its chunk_cumsum listing: the dt tile of one chunk is
    read with zero padding past the sequence end, multiplied by the per-head A,
    summed cumulatively along the chunk (time) axis and scaled by log2(e).
    Returns (cs2, dtT), both (b, H, nc, Q): cs2 the scaled cumsum, dtT the
    zero-padded dt laid out per head, chunk and position.
    """
    dt = np.asarray(dt, np.float64)
    A = np.asarray(A, np.float64)
    b, L, H = dt.shape
    nc = (L + chunk - 1) // chunk
    pad = np.zeros((b, nc * chunk, H))
    pad[:, :L] = dt
    tiles = pad.reshape(b, nc, chunk, H).transpose(0, 3, 1, 2)   # (b, H, nc, Q)
    cs2 = np.cumsum(tiles * A[None, :, None, None], axis=-1) * LOG2E
    return cs2, tiles.copy()


def _expand_groups(M, H):
    G = M.shape[2]
    return M[:, :, np.arange(H) // (H // G)]                 # (b, L, H, N)


def quadratic(x, dt, A, B, C, D=None, init=None):
    """Quadratic (dual, attention-like) form over the whole sequence, float64.

    The matrix form of the same layer that [P1] section 1 and [P3] section 2
    turn into chunked matrix products:  y = (M o (C B^T)) x + exp(cs) C h0^T + D x
    with cs_i = sum_{s<=i} dt_s A and M_ij = exp(cs_i - cs_j) dt_j for j <= i,
    else 0.  O(L^2); for tiny inputs.  Returns (y (b,L,H,P), final (b,H,P,N)).
    """
    x, B, C = widen(x), widen(B), widen(C)
    dt, A = np.asarray(dt, np.float64), np.asarray(A, np.float64)
    b, L, H, P = x.shape
    N = B.shape[3]
    Bh, Ch = _expand_groups(B, H), _expand_groups(C, H)       # (b, L, H, N)
    cs = np.cumsum(dt * A, axis=1)                            # (b, L, H)
    diff = cs[:, :, None, :] - cs[:, None, :, :]              # (b, i, j, H)
    causal = np.tril(np.ones((L, L), dtype=bool))[None, :, :, None]
    M = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0) * dt[:, None, :, :]
    CB = np.einsum("bihn,bjhn->bijh", Ch, Bh)
    y = np.einsum("bijh,bjhp->bihp", M * CB, x)
    h0 = np.zeros((b, H, P, N)) if init is None else np.asarray(init, np.float64)
    y += np.exp(cs)[..., None] * np.einsum("bihn,bhpn->bihp", Ch, h0)
    if D is not None:
        y += np.asarray(D, np.float64)[None, None, :, None] * x
    wlast = np.exp(cs[:, -1:, :] - cs) * dt                   # (b, L, H)
    final = np.einsum("bjh,bjhp,bjhn->bhpn", wlast, x, Bh) + np.exp(cs[:, -1])[..., None, None] * h0
    return y, final


def chunked(x, dt, A, B, C, D=None, init=None, chunk=64):
    """Independent chunked (SSD) evaluation with batched einsums, float64.

    [P3] technical summary section 2: split the sequence into fixed-size
    chunks, express the work as batched einsums with static causal masks, and
    carry the decay in wide precision; [P1] section 2: in-chunk cumsum, the
    state entering each chunk (scanned in chunk order) and the outputs from it.
    Steps: (1) cs = in-chunk cumsum of dt*A; (2) diagonal block outputs
    (L o C B^T) x with L_ij = exp(cs_i - cs_j) dt_j, j <= i; (3) chunk end
    states from zero, sum_j exp(cs_last - cs_j) dt_j x_j (x) B_j; (4) states
    entering each chunk by the sequential chunk scan h <- exp(cs_last) h + S;
    (5) off-diagonal outputs exp(cs_i) C_i . h_in; (6) y = (2) + (5) + D x.
    Returns (y (b,L,H,P), final (b,H,P,N), chunk_in (b,nc,H,P,N), S (b,nc,H,P,N)).
    """
    x, B, C = widen(x), widen(B), widen(C)
    dt, A = np.asarray(dt, np.float64), np.asarray(A, np.float64)
    b, L, H, P = x.shape
    N = B.shape[3]
    Q = chunk
    nc = (L + Q - 1) // Q
    Lp = nc * Q

    def padded(a):
        out = np.zeros((a.shape[0], Lp) + a.shape[2:])
        out[:, :L] = a
        return out.reshape((a.shape[0], nc, Q) + a.shape[2:])

    xc = padded(x)                                           # (b, nc, Q, H, P)
    dtc = padded(dt)                                         # (b, nc, Q, H)
    Bc = padded(_expand_groups(B, H))                        # (b, nc, Q, H, N)
    Cc = padded(_expand_groups(C, H))
    cs = np.cumsum(dtc * A, axis=2)                          # (1)
    seg = cs[:, :, :, None, :] - cs[:, :, None, :, :]        # (b, nc, i, j, H)
    mask = np.tril(np.ones((Q, Q), dtype=bool))[None, None, :, :, None]
    Lm = np.where(mask, np.exp(np.where(mask, seg, 0.0)), 0.0) * dtc[:, :, None, :, :]
    y_diag = np.einsum("bcihn,bcjhn,bcijh,bcjhp->bcihp", Cc, Bc, Lm, xc)           # (2)
    wst = np.exp(cs[:, :, -1:, :] - cs) * dtc                # (b, nc, Q, H)
    S = np.einsum("bcjh,bcjhp,bcjhn->bchpn", wst, xc, Bc)                          # (3)
    h = np.zeros((b, H, P, N)) if init is None else np.asarray(init, np.float64).copy()
    chunk_in = np.empty((b, nc, H, P, N))
    for c in range(nc):                                                           # (4)
        chunk_in[:, c] = h
        h = np.exp(cs[:, c, -1])[..., None, None] * h + S[:, c]
    y_off = np.einsum("bcihn,bchpn,bcih->bcihp", Cc, chunk_in, np.exp(cs))         # (5)
    y = (y_diag + y_off).reshape(b, Lp, H, P)[:, :L]
    if D is not None:
        y = y + np.asarray(D, np.float64)[None, None, :, None] * x                 # (6)
    return y, h, chunk_in, S


def rel_err(got, ref) -> float:
    """max |got - ref| / max |ref| over the whole tensor (the parity metric)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    denom = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if denom == 0.0:
        return 0.0 if num == 0.0 else math.inf
    return num / denom
