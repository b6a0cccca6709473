"""Parity of the decode (recurrent form) entry point with the float64 oracle.

ssd_decode advances a float32 state over a few tokens per launch.  Its y is compared with the
oracle recurrence element by element (bounds: 1e-5 for float32 I/O, 1e-2 for bf16 y, whose
only extra error is the final rounding to bf16), its state after the run with the oracle's
final state (1e-5; the state never leaves float32).  Metric: max|got - ref| / max|ref|.
"""
import numpy as np
import pytest

from oracle import ref
from state_space_model_02_gb300 import ssd, synth

from util import rel, to_device, y_to_numpy

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

Y_TOL = {"f32": 1e-5, "bf16": 1e-2}
STATE_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_02_gb300 import build as cuda_build

    cuda_build.build()
    ssd.load_library()


def run_decode(inp):
    t = to_device(inp)
    state = t["init"].clone() if t["init"] is not None else torch.zeros(
        inp.x.shape[0], inp.x.shape[2], inp.x.shape[3], inp.B.shape[3], device="cuda")
    y = ssd.decode(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], state)
    torch.cuda.synchronize()
    return y_to_numpy(y), state.cpu().numpy()


def oracle(inp):
    out = ref.recurrence(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, chunk=64)
    b, L, H, P = inp.x.shape
    y = out["y"].reshape(b, H, L, P).transpose(0, 2, 1, 3)
    fin = out["final"].reshape(b, H, P, -1)
    return y, fin


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [1, 3, 7, 16])
@pytest.mark.parametrize("N", [64, 128, 256])
def test_decode_matches_oracle(dtype, T, N):
    inp = synth.make_inputs(batch=3, seqlen=T, nheads=5, headdim=64, dstate=N, io_dtype=dtype,
                            init=True, seed=21 + T + N)
    y, st = run_decode(inp)
    y_ref, st_ref = oracle(inp)
    assert rel(y, y_ref) <= Y_TOL[dtype]
    assert rel(st, st_ref) <= STATE_TOL


def test_decode_groups_no_D_zero_state():
    inp = synth.make_inputs(batch=2, seqlen=4, nheads=8, headdim=64, dstate=128, ngroups=4,
                            io_dtype="bf16", init=False, seed=31, with_D=False)
    y, st = run_decode(inp)
    y_ref, st_ref = oracle(inp)
    assert rel(y, y_ref) <= Y_TOL["bf16"]
    assert rel(st, st_ref) <= STATE_TOL


def test_decode_state_size_512():
    inp = synth.make_inputs(batch=1, seqlen=2, nheads=3, headdim=64, dstate=512, io_dtype="bf16",
                            init=True, seed=33)
    y, st = run_decode(inp)
    y_ref, st_ref = oracle(inp)
    assert rel(y, y_ref) <= Y_TOL["bf16"]
    assert rel(st, st_ref) <= STATE_TOL


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_state_size_1024_per_head_kernel(dtype):
    # N = 1024 is beyond the row-streaming kernel's sizes: the per-head kernel serves it
    inp = synth.make_inputs(batch=2, seqlen=5, nheads=3, headdim=16, dstate=1024, io_dtype=dtype,
                            init=True, seed=35)
    y, st = run_decode(inp)
    y_ref, st_ref = oracle(inp)
    assert rel(y, y_ref) <= Y_TOL[dtype]
    assert rel(st, st_ref) <= STATE_TOL


def test_decode_many_heads_partial_last_block():
    # 1 x 3 heads x (16 x 128) floats = 6 warps of 1024 floats in the row-streaming kernel:
    # the second block of four warps is half empty
    inp = synth.make_inputs(batch=1, seqlen=9, nheads=3, headdim=16, dstate=128, io_dtype="bf16",
                            init=True, seed=37)
    y, st = run_decode(inp)
    y_ref, st_ref = oracle(inp)
    assert rel(y, y_ref) <= Y_TOL["bf16"]
    assert rel(st, st_ref) <= STATE_TOL


def test_multi_token_launch_equals_single_token_launches():
    inp = synth.make_inputs(batch=2, seqlen=8, nheads=4, headdim=64, dstate=128, io_dtype="bf16",
                            init=True, seed=41)
    t = to_device(inp)
    state_a = t["init"].clone()
    y_a = ssd.decode(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], state_a)
    state_b = t["init"].clone()
    ys = []
    for k in range(8):
        sl = slice(k, k + 1)
        ys.append(ssd.decode(t["x"][:, sl].contiguous(), t["dt"][:, sl].contiguous(), t["A"],
                             t["B"][:, sl].contiguous(), t["C"][:, sl].contiguous(), t["D"], state_b))
    torch.cuda.synchronize()
    assert torch.equal(y_a, torch.cat(ys, dim=1))
    assert torch.equal(state_a, state_b)


def test_decode_continues_a_prefill():
    # prefill L tokens with the chunked scan, then decode T more from its final state
    L, T = 512, 6
    inp = synth.make_inputs(batch=2, seqlen=L + T, nheads=4, headdim=64, dstate=128,
                            io_dtype="bf16", init=True, seed=43)
    t = to_device(inp)
    pre = slice(0, L)
    _, state = ssd.fwd(t["x"][:, pre].contiguous(), t["dt"][:, pre].contiguous(), t["A"],
                       t["B"][:, pre].contiguous(), t["C"][:, pre].contiguous(), t["D"], chunk=256,
                       init_state=t["init"])
    dec = slice(L, L + T)
    y = ssd.decode(t["x"][:, dec].contiguous(), t["dt"][:, dec].contiguous(), t["A"],
                   t["B"][:, dec].contiguous(), t["C"][:, dec].contiguous(), t["D"], state)
    torch.cuda.synchronize()
    y_ref, st_ref = oracle(inp)
    assert rel(y_to_numpy(y), y_ref[:, L:]) <= 2e-2
    assert rel(state.cpu().numpy(), st_ref) <= 2e-2
