"""ssd_fwd_noalloc: the forward pass for callers that cannot allocate device memory.

Some callers of this library cannot obtain device scratch memory at all -- a plugin inside
a host application that owns the device-memory budget, or a serving loop that must never
enter the allocator.  ssd_fwd_noalloc takes its scratch from a fixed array in the library's
device image instead of a caller workspace.  These tests call it through the C ABI and
check its results against ssd_fwd (the entry point with a caller workspace) on the same
inputs, for two calls in a row whose shapes differ, so the second call runs on an array
still holding the first call's intermediates.  Both entry points run the same deterministic
kernels, so the results must agree bit for bit.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

from state_space_model_02_gb300 import ssd, synth

from util import to_device, y_to_numpy

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NOALLOC_MAX = 64 << 20   # SSD_NOALLOC_MAX_WORKSPACE_BYTES in include/ssd.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_02_gb300 import build as cuda_build

    cuda_build.build()
    return ssd.load_library()


def _noalloc(lib, t, prob):
    y = torch.full_like(t["x"], float("nan"))
    fin = torch.full((prob.batch, prob.nheads, prob.headdim, prob.dstate), float("nan"),
                     dtype=torch.float32, device="cuda")
    p = ssd._p
    rc = lib.ssd_fwd_noalloc(ctypes.byref(prob.c_shape()), p(t["x"]), p(t["dt"]), p(t["A"]), p(t["B"]),
                             p(t["C"]), p(t["D"]), p(t["init"]), p(y), p(fin),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, y, fin


def _with_workspace(t, chunk):
    y, fin = ssd.fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], chunk=chunk, init_state=t["init"])
    return y, fin


CASES = [
    dict(name="mamba2_130m_layer"),   # about 25.5 MiB of scratch
    dict(shape=dict(batch=1, seqlen=1000, nheads=6, headdim=64, dstate=128, chunk=256,
                    io_dtype="bf16", init=True), seed=4),
]


def _inputs(case):
    if "name" in case:
        return synth.make_config(case["name"], seed=1)
    return synth.make_inputs(seed=case["seed"], **case["shape"])


def test_two_calls_in_a_row_match_the_workspace_entry_point(lib):
    for case in CASES:
        inp = _inputs(case)
        t = to_device(inp)
        prob = ssd.problem_of(t["x"], t["B"], inp.chunk)
        assert ssd.workspace_bytes(prob) <= NOALLOC_MAX
        rc, y, fin = _noalloc(lib, t, prob)
        assert rc == 0, lib.ssd_last_error()
        y_ref, fin_ref = _with_workspace(t, inp.chunk)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        assert torch.equal(fin, fin_ref)
        assert np.isfinite(y_to_numpy(y)).all()


def test_shapes_beyond_the_fixed_array_are_rejected_without_launching(lib):
    inp = synth.make_inputs(batch=1, seqlen=16384, nheads=32, headdim=64, dstate=128, chunk=256,
                            io_dtype="bf16", init=False, seed=2)   # needs about 101 MiB
    t = to_device(inp)
    prob = ssd.problem_of(t["x"], t["B"], inp.chunk)
    assert ssd.workspace_bytes(prob) > NOALLOC_MAX
    rc, y, fin = _noalloc(lib, t, prob)
    torch.cuda.synchronize()
    assert rc == 6                                   # SSD_ERR_WORKSPACE
    assert b"workspace" in lib.ssd_last_error()
    assert torch.isnan(y.float()).all() and torch.isnan(fin).all()   # nothing was written
