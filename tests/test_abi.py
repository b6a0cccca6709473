"""C-ABI boundary checks that need no GPU: the library builds, loads and exports every
entry point include/ssd.h declares, and host-side validation rejects bad arguments before
any CUDA call."""
import ctypes
import os
import re

import pytest

from state_space_model_02_gb300 import build as cuda_build
from state_space_model_02_gb300 import ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return ssd.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "ssd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(ssd_[a-z_]+)\s*\(", text, flags=re.M)


def test_header_declares_the_binding_exports():
    assert tuple(header_functions()) == ssd.EXPORTS


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr), name


def test_missing_library_fails_loudly(tmp_path):
    saved = ssd._lib
    ssd._lib = None
    try:
        with pytest.raises(RuntimeError):
            ssd.load_library(str(tmp_path / "libssd.so"))
    finally:
        ssd._lib = saved


def shape(**kw):
    base = dict(batch=2, seqlen=8192, nheads=80, headdim=64, dstate=128, ngroups=1, chunk=256,
                io_dtype=ssd.SSD_BF16, flags=0)
    base.update(kw)
    return ssd.Problem(**base)


def test_workspace_size_and_layout(lib):
    p = shape()
    n = ssd.workspace_bytes(p)
    lay = ssd.workspace_layout(p)
    nc = 32
    assert lay.nchunks == nc and lay.total == n
    assert lay.cs2 % 1024 == 0 and lay.dtT % 1024 == 0 and lay.S % 1024 == 0 and lay.hprev % 1024 == 0
    assert lay.dtT - lay.cs2 >= 2 * 80 * nc * 256 * 4
    assert lay.hprev - lay.S >= 2 * nc * 80 * 64 * 128 * 2   # S in the bf16 I/O dtype
    assert n - lay.hprev >= 2 * nc * 80 * 64 * 128 * 2
    # ragged length rounds the chunk count up
    assert ssd.workspace_layout(shape(seqlen=8193)).nchunks == 33


@pytest.mark.parametrize("bad", [dict(chunk=100), dict(nheads=81, ngroups=2), dict(batch=0),
                                 dict(io_dtype=7), dict(seqlen=0)])
def test_invalid_shapes_are_rejected(lib, bad):
    s = shape(**bad).c_shape()
    assert lib.ssd_workspace_bytes(ctypes.byref(s)) == 0
    rc = lib.ssd_fwd(ctypes.byref(s), *([ctypes.c_void_p(0x10000)] * 10), 1 << 40, None)
    assert rc == 1 and lib.ssd_last_error()


def test_null_and_misaligned_pointers_are_rejected_before_any_launch(lib):
    s = shape().c_shape()
    good = ctypes.c_void_p(0x100000)
    args = [good] * 10
    # null x
    a = list(args)
    a[0] = None
    assert lib.ssd_fwd(ctypes.byref(s), *a, 1 << 40, None) == 1
    # misaligned B
    a = list(args)
    a[3] = ctypes.c_void_p(0x100008)
    assert lib.ssd_fwd(ctypes.byref(s), *a, 1 << 40, None) == 3
    # missing workspace / too small workspace
    a = list(args)
    a[9] = None
    assert lib.ssd_fwd(ctypes.byref(s), *a, 1 << 40, None) == 6
    assert lib.ssd_fwd(ctypes.byref(s), *args, 1024, None) == 6
    assert b"workspace" in lib.ssd_last_error()


def test_status_strings(lib):
    for code in range(7):
        assert lib.ssd_status_str(code)
    assert lib.ssd_status_str(5) == b"on-chip wait timed out"


def test_require_tensor_cores_rejects_fallback_shapes_before_launch(lib):
    # no GPU needed: the check happens on the host before the workspace is even looked at
    for kw, why in [(dict(headdim=32), b"headdim"), (dict(chunk=64), b"chunk"), (dict(io_dtype=0), b"float32"),
                    (dict(dstate=48), b"dstate")]:
        s = shape(flags=ssd.FLAG_REQUIRE_TENSOR_CORES, **kw).c_shape()
        rc = lib.ssd_fwd(ctypes.byref(s), *([ctypes.c_void_p(16)] * 10), 0, None)
        assert rc == 2 and why in lib.ssd_last_error(), (kw, rc, lib.ssd_last_error())
    # a tensor-core shape passes that check and fails later, on the (missing) workspace
    s = shape(flags=ssd.FLAG_REQUIRE_TENSOR_CORES).c_shape()
    assert lib.ssd_fwd(ctypes.byref(s), *([ctypes.c_void_p(16)] * 10), 0, None) == 6


def test_kernel_plan(lib):
    assert ssd.kernel_plan(shape()) == 3                              # both steps on tensor cores
    assert ssd.kernel_plan(shape(batch=4, seqlen=2048, nheads=24)) == 3
    assert ssd.kernel_plan(shape(dstate=256)) & 2                     # wide tensor-core chunk_scan
    assert ssd.kernel_plan(shape(dstate=384)) & 2
    assert ssd.kernel_plan(shape(dstate=512)) & 2
    assert ssd.kernel_plan(shape(dstate=640)) & 2
    assert ssd.kernel_plan(shape(dstate=192, chunk=128)) & 2
    assert not ssd.kernel_plan(shape(dstate=192)) & 2                 # below the 256-token chunk
    assert not ssd.kernel_plan(shape(dstate=200)) & 2                 # not a multiple of 64
    assert ssd.kernel_plan(shape(flags=ssd.FLAG_FORCE_SIMT)) == 0
    assert ssd.kernel_plan(shape(io_dtype=ssd.SSD_F32)) == 0          # exact-fp32 CUDA-core path
    assert ssd.kernel_plan(shape(headdim=32)) == 0
    assert ssd.kernel_plan(shape(chunk=64)) == 0
    assert ssd.kernel_plan(shape(chunk=100)) == -1
    # fused fwd_pass_state: only with its flag, where the shape allows it (N <= 128); SEPARATE
    # wins over FUSED
    fused, sep = ssd.FLAG_FUSED_STATE, ssd.FLAG_SEPARATE_STATE_PASSING
    assert ssd.kernel_plan(shape(flags=fused)) == 7
    assert ssd.kernel_plan(shape(dstate=64, flags=fused)) == 7
    assert ssd.kernel_plan(shape(dstate=256, flags=fused)) == 3
    assert ssd.kernel_plan(shape(chunk=64, flags=fused)) == 0
    assert ssd.kernel_plan(shape(flags=fused | sep)) == 3
    assert ssd.kernel_plan(shape()) & 4 == 0


def test_selftest_rejects_bad_limits(lib):
    assert lib.ssd_selftest_wait_timeout(None, 1000, None) == 1
    assert lib.ssd_selftest_wait_timeout(ctypes.c_void_p(0x1000), 0, None) == 1
    assert lib.ssd_selftest_wait_timeout(ctypes.c_void_p(0x1000), 2_000_000_000, None) == 1


def test_decode_rejects_bad_arguments_before_any_launch(lib):
    good = ctypes.c_void_p(0x100000)
    args = [good] * 8
    s = shape(seqlen=1).c_shape()
    # dstate not a multiple of 64
    bad = shape(seqlen=1, dstate=48).c_shape()
    assert lib.ssd_decode(ctypes.byref(bad), *args, None) == 2
    # dstate / 64 not a power of two
    bad = shape(seqlen=1, dstate=192).c_shape()
    assert lib.ssd_decode(ctypes.byref(bad), *args, None) == 2
    # null state
    a = list(args)
    a[6] = None
    assert lib.ssd_decode(ctypes.byref(s), *a, None) == 1
    # misaligned x
    a = list(args)
    a[0] = ctypes.c_void_p(0x100004)
    assert lib.ssd_decode(ctypes.byref(s), *a, None) == 3
    # the chunk field is not used by the recurrent form
    odd = shape(seqlen=1, chunk=100).c_shape()
    assert lib.ssd_decode(ctypes.byref(odd), *([None] * 8), None) == 1  # null x, not the chunk


def test_selective_scan_rejects_bad_arguments_before_any_launch(lib):
    good = ctypes.c_void_p(0x100000)
    args = [good] * 5 + [None, None, None, good]   # x, delta, A, B, C, Dskip, init, final, y

    def sh(**kw):
        base = dict(batch=2, seqlen=64, dim=1536, dstate=16, io_dtype=ssd.SSD_BF16, flags=0)
        base.update(kw)
        return ssd.SelShape(**base)

    assert lib.ssd_selective_scan(None, *args, None) == 1
    assert lib.ssd_selective_scan(ctypes.byref(sh(seqlen=0)), *args, None) == 1
    assert lib.ssd_selective_scan(ctypes.byref(sh(io_dtype=7)), *args, None) == 1
    # state sizes outside {8, 16, 32, 64}; a channel count that does not fill whole warps
    assert lib.ssd_selective_scan(ctypes.byref(sh(dstate=12)), *args, None) == 2
    assert lib.ssd_selective_scan(ctypes.byref(sh(dstate=128)), *args, None) == 2
    assert lib.ssd_selective_scan(ctypes.byref(sh(dim=1538)), *args, None) == 2
    a = list(args)
    a[0] = None
    assert lib.ssd_selective_scan(ctypes.byref(sh()), *a, None) == 1
    a = list(args)
    a[3] = ctypes.c_void_p(0x100008)
    assert lib.ssd_selective_scan(ctypes.byref(sh()), *a, None) == 3
    a = list(args)
    a[6] = ctypes.c_void_p(0x100004)   # misaligned init_state
    assert lib.ssd_selective_scan(ctypes.byref(sh()), *a, None) == 3
