"""Parity of the Mamba-1 selective scan (ssd_selective_scan) with the float64 oracle.

Metric: max|got - ref| / max|ref| over the compared tensor.  Bounds: y 1e-4 for float32 I/O
and 2e-2 for bf16 I/O (whose y is rounded to bf16 once); final state 1e-4 in both (it never
leaves float32).  Shapes cover every supported state size, ragged token blocks (the kernel
stages 32 tokens at a time and reduces N/2 tokens at a time), A = 0 entries (the limit of the
zero-order hold), large |delta A| (the other branch of the hold's factor), no skip, no init,
and the full Mamba-1 130M / 2.8B layer shapes on sampled channels.
"""
import numpy as np
import pytest

from oracle import selective as sel
from state_space_model_02_gb300 import ssd, synth

from util import rel, y_to_numpy

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

Y_TOL = {"f32": 1e-4, "bf16": 2e-2}
STATE_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_02_gb300 import build as cuda_build

    cuda_build.build()
    ssd.load_library()


def dev(inp):
    bf16 = inp.io_dtype == "bf16"

    def io(a):
        if bf16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dict(x=io(inp.x), delta=io(inp.delta), A=f32(inp.A), B=io(inp.B), C=io(inp.C), D=f32(inp.D),
                init=f32(inp.init))


def run(inp, **kw):
    t = dev(inp)
    y, fin = ssd.selective_scan(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["init"], **kw)
    torch.cuda.synchronize()
    return y_to_numpy(y), fin.cpu().numpy()


def check(inp):
    y, fin = run(inp)
    o = sel.selective_scan(inp.x, inp.delta, inp.A, inp.B, inp.C, inp.D, inp.init)
    assert rel(y, o["y"]) <= Y_TOL[inp.io_dtype]
    assert rel(fin, o["final"]) <= STATE_TOL


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [8, 16, 32, 64])
def test_matches_oracle(dtype, N):
    D = 3 * (64 // N) * 2
    check(synth.make_selective_inputs(2, 67, D, N, io_dtype=dtype, init=True, seed=100 + N))


@pytest.mark.parametrize("L", [1, 5, 32, 33, 100])
def test_ragged_lengths(L):
    check(synth.make_selective_inputs(1, L, 16, 16, io_dtype="f32", init=True, seed=200 + L))


def test_no_skip_no_init():
    check(synth.make_selective_inputs(2, 45, 32, 16, io_dtype="bf16", init=False, with_D=False, seed=301))


def test_zero_A_entries_take_the_limit():
    inp = synth.make_selective_inputs(1, 70, 8, 16, io_dtype="f32", init=True, seed=303)
    inp.A[:, ::3] = 0.0
    inp.A[2, :] = 0.0
    check(inp)


def test_large_delta_A_branch():
    # |delta A| up to 0.1 * 400 = 40: the (exp(w) - 1) / A form of the hold's factor
    check(synth.make_selective_inputs(1, 64, 16, 16, io_dtype="f32", init=True, a_range=(0.5, 400.0), seed=305))


def test_split_and_resume_is_exact():
    inp = synth.make_selective_inputs(2, 96, 24, 16, io_dtype="bf16", init=True, seed=307)
    t = dev(inp)
    y, fin = ssd.selective_scan(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["init"])
    k = 40
    part = lambda a, s: a[:, s].contiguous()
    y1, f1 = ssd.selective_scan(part(t["x"], slice(0, k)), part(t["delta"], slice(0, k)), t["A"],
                                part(t["B"], slice(0, k)), part(t["C"], slice(0, k)), t["D"], t["init"])
    y2, f2 = ssd.selective_scan(part(t["x"], slice(k, None)), part(t["delta"], slice(k, None)), t["A"],
                                part(t["B"], slice(k, None)), part(t["C"], slice(k, None)), t["D"], f1)
    torch.cuda.synchronize()
    assert torch.equal(y, torch.cat([y1, y2], dim=1))
    assert torch.equal(fin, f2)


@pytest.mark.parametrize("name,nch", [("mamba1_130m_layer", 48), ("mamba1_2p8b_layer", 40)])
def test_full_layer_sampled_channels(name, nch):
    inp = synth.make_selective_config(name)
    y, fin = run(inp)
    rng = np.random.default_rng(1)
    D = inp.x.shape[2]
    ch = np.unique(np.concatenate([[0, D - 1], rng.choice(D, nch, replace=False)]))
    sub = lambda a: np.ascontiguousarray(a[:, :, ch])
    o = sel.selective_scan(sub(inp.x), sub(inp.delta), inp.A[ch], inp.B, inp.C, inp.D[ch],
                           None if inp.init is None else np.ascontiguousarray(inp.init[:, ch]))
    assert rel(y[:, :, ch], o["y"]) <= Y_TOL[inp.io_dtype]
    assert rel(fin[:, ch], o["final"]) <= STATE_TOL
