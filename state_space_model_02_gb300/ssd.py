"""Python binding of libssd.so (include/ssd.h): argument marshalling only.

Every step of the forward scan runs in the library's CUDA kernels; PyTorch only
provides device memory and the current stream.  If the library is missing the
first call raises -- there is no fallback.
"""
import ctypes
import os
import warnings
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libssd.so")

SSD_F32, SSD_BF16 = 0, 1
FLAG_FORCE_SIMT = 1
FLAG_REQUIRE_TENSOR_CORES = 2   # fail (SSD_ERR_UNSUPPORTED) rather than fall back to the CUDA cores
FLAG_SEPARATE_STATE_PASSING = 4  # chunk_state and state_passing as two kernels (the default)
FLAG_FUSED_STATE = 8             # the fused fwd_pass_state kernel wherever the shape allows it
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_ALIGN",
          4: "SSD_ERR_CUDA", 5: "SSD_ERR_TIMEOUT", 6: "SSD_ERR_WORKSPACE"}

# Every entry point of include/ssd.h, in declaration order.
EXPORTS = ("ssd_workspace_bytes", "ssd_get_workspace_layout", "ssd_fwd", "ssd_chunk_cumsum",
           "ssd_chunk_state", "ssd_state_passing", "ssd_fwd_pass_state", "ssd_chunk_scan", "ssd_read_status",
           "ssd_selftest_wait_timeout", "ssd_fwd_noalloc", "ssd_decode", "ssd_selective_scan",
           "ssd_bwd_workspace_bytes", "ssd_bwd",
           "ssd_status_str", "ssd_last_error", "ssd_kernel_plan")


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk", ctypes.c_int64), ("io_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class SelShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("dim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("io_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [("status", ctypes.c_size_t), ("cs2", ctypes.c_size_t), ("dtT", ctypes.c_size_t),
                ("S", ctypes.c_size_t), ("hprev", ctypes.c_size_t), ("total", ctypes.c_size_t),
                ("nchunks", ctypes.c_int64)]


class SSDError(RuntimeError):
    def __init__(self, status, detail=""):
        self.status = status
        super().__init__("%s: %s" % (STATUS.get(status, str(status)), detail))


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libssd.so and declare its signatures (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libssd.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    vp, sp = ctypes.c_void_p, ctypes.POINTER(Shape)
    sig = {
        "ssd_workspace_bytes": ([sp], ctypes.c_size_t),
        "ssd_get_workspace_layout": ([sp, ctypes.POINTER(WorkspaceLayout)], ctypes.c_int),
        "ssd_fwd": ([sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "ssd_chunk_cumsum": ([sp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "ssd_chunk_state": ([sp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "ssd_state_passing": ([sp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "ssd_fwd_pass_state": ([sp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "ssd_chunk_scan": ([sp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "ssd_read_status": ([vp, vp], ctypes.c_int),
        "ssd_selftest_wait_timeout": ([vp, ctypes.c_uint64, vp], ctypes.c_int),
        "ssd_fwd_noalloc": ([sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "ssd_decode": ([sp, vp, vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "ssd_selective_scan": ([ctypes.POINTER(SelShape)] + [vp] * 10, ctypes.c_int),
        "ssd_bwd_workspace_bytes": ([sp], ctypes.c_size_t),
        "ssd_bwd": ([sp] + [vp] * 17 + [ctypes.c_size_t, vp], ctypes.c_int),
        "ssd_status_str": ([ctypes.c_int], ctypes.c_char_p),
        "ssd_last_error": ([], ctypes.c_char_p),
        "ssd_kernel_plan": ([sp], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(rc):
    if rc != 0:
        raise SSDError(rc, load_library().ssd_last_error().decode())


@dataclass
class Problem:
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int = 1
    chunk: int = 256
    io_dtype: int = SSD_BF16
    flags: int = 0

    def c_shape(self) -> Shape:
        return Shape(self.batch, self.seqlen, self.nheads, self.headdim, self.dstate, self.ngroups,
                     self.chunk, self.io_dtype, self.flags)


def _torch():
    import torch  # PyTorch is device-memory and stream plumbing only
    return torch


def problem_of(x, B, chunk, flags=0) -> Problem:
    torch = _torch()
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if x.dtype == torch.bfloat16:
        io = SSD_BF16
    elif x.dtype == torch.float32:
        io = SSD_F32
    else:
        raise TypeError("x must be bfloat16 or float32")
    return Problem(b, L, H, P, N, G, chunk, io, flags)


def workspace_bytes(prob: Problem) -> int:
    n = load_library().ssd_workspace_bytes(ctypes.byref(prob.c_shape()))
    if n == 0:
        raise SSDError(1, load_library().ssd_last_error().decode())
    return int(n)


def workspace_layout(prob: Problem) -> WorkspaceLayout:
    out = WorkspaceLayout()
    _check(load_library().ssd_get_workspace_layout(ctypes.byref(prob.c_shape()), ctypes.byref(out)))
    return out


_fallback_warned = set()


def _warn_cuda_cores(prob: Problem):
    """Warns once per shape when bf16 work falls back to the float32 CUDA-core kernels."""
    if prob.io_dtype != SSD_BF16 or prob.flags & (FLAG_FORCE_SIMT | FLAG_REQUIRE_TENSOR_CORES):
        return
    key = (prob.headdim, prob.dstate, prob.chunk)
    if key in _fallback_warned or kernel_plan(prob) & 3 == 3:
        return
    _fallback_warned.add(key)
    warnings.warn("ssd.fwd: headdim %d, dstate %d, chunk %d run chunk_state / chunk_scan on the "
                  "CUDA cores (tensor-core plan %d of 3); pass flags=FLAG_REQUIRE_TENSOR_CORES to "
                  "make this an error" % (prob.headdim, prob.dstate, prob.chunk, kernel_plan(prob) & 3),
                  RuntimeWarning, stacklevel=3)


def kernel_plan(prob: Problem) -> int:
    """bit 0: chunk_state on tensor cores, bit 1: chunk_scan on tensor cores, bit 2: the fused
    fwd_pass_state kernel (chunk_state + state_passing in one; with FLAG_FUSED_STATE)."""
    return int(load_library().ssd_kernel_plan(ctypes.byref(prob.c_shape())))


def alloc_workspace(prob: Problem, device="cuda"):
    torch = _torch()
    return torch.empty(workspace_bytes(prob), dtype=torch.uint8, device=device)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype=None, shape=None):
    torch = _torch()
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s" % (name, dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def fwd(x, dt, A, B, C, D=None, chunk=256, init_state=None, *, y=None, final_state=None,
        want_final=True, workspace=None, stream=None, flags=0):
    """ssd_fwd: returns (y, final_state).  All tensors on the same CUDA device.

    x (b,L,H,P) and B, C (b,L,G,N) in bf16 or fp32 (one dtype); dt (b,L,H), A (H),
    D (H), init_state (b,H,P,N) in fp32.  ``workspace`` (uint8, >= workspace_bytes)
    is allocated when absent.  Work is enqueued on ``stream`` (default: current).
    """
    torch = _torch()
    prob = problem_of(x, B, chunk, flags)
    b, L, H, P, N, G = prob.batch, prob.seqlen, prob.nheads, prob.headdim, prob.dstate, prob.ngroups
    _warn_cuda_cores(prob)
    _need(x, "x", x.dtype)
    _need(B, "B", x.dtype, (b, L, G, N))
    _need(C, "C", x.dtype, (b, L, G, N))
    _need(dt, "dt", torch.float32, (b, L, H))
    _need(A, "A", torch.float32, (H,))
    _need(D, "D", torch.float32, (H,))
    _need(init_state, "init_state", torch.float32, (b, H, P, N))
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", x.dtype, x.shape)
    if final_state is None and want_final:
        final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(prob, x.device)
    rc = load_library().ssd_fwd(ctypes.byref(prob.c_shape()), _p(x), _p(dt), _p(A), _p(B), _p(C),
                                _p(D), _p(init_state), _p(y), _p(final_state), _p(workspace),
                                workspace.numel(), _stream(stream))
    _check(rc)
    return y, final_state


def decode(x, dt, A, B, C, D, state, *, y=None, stream=None):
    """ssd_decode: advances ``state`` (fp32, (b,H,P,N), updated in place) over the L tokens of
    x (b,L,H,P) and returns y (b,L,H,P).  B, C (b,L,G,N) in x's dtype; dt (b,L,H), A and D (H)
    in fp32.  Work is enqueued on ``stream`` (default: current).
    """
    torch = _torch()
    prob = problem_of(x, B, 64)
    b, L, H, P, N, G = prob.batch, prob.seqlen, prob.nheads, prob.headdim, prob.dstate, prob.ngroups
    _need(x, "x", x.dtype)
    _need(B, "B", x.dtype, (b, L, G, N))
    _need(C, "C", x.dtype, (b, L, G, N))
    _need(dt, "dt", torch.float32, (b, L, H))
    _need(A, "A", torch.float32, (H,))
    _need(D, "D", torch.float32, (H,))
    _need(state, "state", torch.float32, (b, H, P, N))
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", x.dtype, x.shape)
    _check(load_library().ssd_decode(ctypes.byref(prob.c_shape()), _p(x), _p(dt), _p(A), _p(B), _p(C),
                                      _p(D), _p(state), _p(y), _stream(stream)))
    return y


def selective_scan(x, delta, A, B, C, Dskip=None, init_state=None, *, y=None, final_state=None,
                   want_final=True, stream=None):
    """ssd_selective_scan (Mamba-1): returns (y, final_state or None).

    x, delta (b,L,D) and B, C (b,L,N) in one dtype (bf16 or fp32); A (D,N), Dskip (D) and
    init_state (b,D,N) in fp32.  Work is enqueued on ``stream`` (default: current).
    """
    torch = _torch()
    if x.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be (b, L, D) and B (b, L, N)")
    b, L, D = x.shape
    N = B.shape[2]
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be bfloat16 or float32")
    _need(x, "x", x.dtype)
    _need(delta, "delta", x.dtype, (b, L, D))
    _need(B, "B", x.dtype, (b, L, N))
    _need(C, "C", x.dtype, (b, L, N))
    _need(A, "A", torch.float32, (D, N))
    _need(Dskip, "Dskip", torch.float32, (D,))
    _need(init_state, "init_state", torch.float32, (b, D, N))
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", x.dtype, x.shape)
    if final_state is None and want_final:
        final_state = torch.empty((b, D, N), dtype=torch.float32, device=x.device)
    _need(final_state, "final_state", torch.float32, (b, D, N))
    shape = SelShape(b, L, D, N, SSD_BF16 if x.dtype == torch.bfloat16 else SSD_F32, 0)
    _check(load_library().ssd_selective_scan(ctypes.byref(shape), _p(x), _p(delta), _p(A), _p(B), _p(C),
                                             _p(Dskip), _p(init_state), _p(final_state), _p(y),
                                             _stream(stream)))
    return y, final_state


def bwd(x, dt, A, B, C, D, dy, chunk=256, init_state=None, dfinal=None, *, workspace=None, stream=None,
        flags=0):
    """ssd_bwd: gradients of the forward scan given dy (and dfinal).  Returns a dict with
    dx, ddt, dA, dB, dC, dD and dinit (None when init_state is None)."""
    torch = _torch()
    prob = problem_of(x, B, chunk, flags)
    b, L, H, P, N, G = prob.batch, prob.seqlen, prob.nheads, prob.headdim, prob.dstate, prob.ngroups
    _warn_cuda_cores(prob)
    _need(x, "x", x.dtype)
    _need(B, "B", x.dtype, (b, L, G, N))
    _need(C, "C", x.dtype, (b, L, G, N))
    _need(dy, "dy", x.dtype, x.shape)
    _need(dt, "dt", torch.float32, (b, L, H))
    _need(A, "A", torch.float32, (H,))
    _need(D, "D", torch.float32, (H,))
    _need(init_state, "init_state", torch.float32, (b, H, P, N))
    _need(dfinal, "dfinal", torch.float32, (b, H, P, N))
    lib = load_library()
    nbytes = lib.ssd_bwd_workspace_bytes(ctypes.byref(prob.c_shape()))
    if nbytes == 0:
        raise SSDError(1, "bad shape")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    out = dict(dx=torch.empty_like(x), ddt=torch.empty_like(dt), dA=torch.empty_like(A), dB=torch.empty_like(B),
               dC=torch.empty_like(C), dD=torch.empty(H, dtype=torch.float32, device=x.device),
               dinit=None if init_state is None else torch.empty_like(init_state))
    _check(lib.ssd_bwd(ctypes.byref(prob.c_shape()), _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(init_state),
                       _p(dy), _p(dfinal), _p(out["dx"]), _p(out["ddt"]), _p(out["dA"]), _p(out["dB"]),
                       _p(out["dC"]), _p(out["dD"]), _p(out["dinit"]), _p(workspace), workspace.numel(),
                       _stream(stream)))
    return out


def chunk_cumsum(prob, dt, A, workspace, stream=None):
    _check(load_library().ssd_chunk_cumsum(ctypes.byref(prob.c_shape()), _p(dt), _p(A), _p(workspace),
                                           workspace.numel(), _stream(stream)))


def chunk_state(prob, x, B, workspace, stream=None):
    _check(load_library().ssd_chunk_state(ctypes.byref(prob.c_shape()), _p(x), _p(B), _p(workspace),
                                          workspace.numel(), _stream(stream)))


def state_passing(prob, init_state, final_state, workspace, stream=None):
    _check(load_library().ssd_state_passing(ctypes.byref(prob.c_shape()), _p(init_state),
                                            _p(final_state), _p(workspace), workspace.numel(),
                                            _stream(stream)))


def fwd_pass_state(prob, x, B, init_state, final_state, workspace, stream=None):
    """chunk_state + state_passing: one fused kernel where it applies, else the two steps."""
    _check(load_library().ssd_fwd_pass_state(ctypes.byref(prob.c_shape()), _p(x), _p(B), _p(init_state),
                                             _p(final_state), _p(workspace), workspace.numel(),
                                             _stream(stream)))


def chunk_scan(prob, x, B, C, D, y, workspace, stream=None):
    _check(load_library().ssd_chunk_scan(ctypes.byref(prob.c_shape()), _p(x), _p(B), _p(C), _p(D),
                                         _p(y), _p(workspace), workspace.numel(), _stream(stream)))


def read_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the workspace status word as an ssd_status."""
    return int(load_library().ssd_read_status(_p(workspace), _stream(stream)))


def selftest_wait_timeout(status_word, timeout_ns, stream=None):
    _check(load_library().ssd_selftest_wait_timeout(_p(status_word), int(timeout_ns), _stream(stream)))


def intermediates(prob: Problem, workspace):
    """Views (cs2, dtT, S, hprev) into a workspace after a forward pass."""
    torch = _torch()
    lay = workspace_layout(prob)
    b, H, P, N, Q, nc = prob.batch, prob.nheads, prob.headdim, prob.dstate, prob.chunk, lay.nchunks

    def view(off, count, dtype, shape):
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return workspace[off:off + nbytes].view(dtype).view(*shape)

    cs2 = view(lay.cs2, b * H * nc * Q, torch.float32, (b, H, nc, Q))
    dtT = view(lay.dtT, b * H * nc * Q, torch.float32, (b, H, nc, Q))
    hdt = torch.bfloat16 if prob.io_dtype == SSD_BF16 else torch.float32
    S = view(lay.S, b * nc * H * P * N, hdt, (b, nc, H, P, N))
    hprev = view(lay.hprev, b * nc * H * P * N, hdt, (b, nc, H, P, N))
    return cs2, dtT, S, hprev
