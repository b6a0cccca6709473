"""Parity of the backward pass (ssd_bwd) with the float64 adjoint oracle (oracle/ref_bwd.py).

Metric per gradient: max|got - ref| / max|ref|.  Bounds: 1e-4 with float32 I/O (every scan runs
in float32 there) and 2e-2 with bf16 I/O, the forward's bounds.  Measured with bf16 on GB300
(the 130M layer, every gradient over the whole tensor): dx 2.8e-3, dB 4.6e-3, dC 3.6e-3,
dA 7.4e-5, ddt 7.1e-6, dD 1.3e-7 -- the two scans that feed ddt and dA run in float32.
"""
import numpy as np
import pytest

from oracle.ref_bwd import recurrence_bwd_np
from state_space_model_02_gb300 import ssd, synth

from util import rel, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_02_gb300 import build as cuda_build

    cuda_build.build()
    ssd.load_library()


def _bf16_bits(a):
    return synth.to_bf16_bits(np.asarray(a, np.float32))


def run_case(dtype, b, L, H, P, N, G, chunk, init=True, with_dfinal=True, seed=0, tol=None, tol_sc=None):
    inp = synth.make_inputs(b, L, H, P, N, G, chunk=chunk, io_dtype=dtype, init=init, seed=seed)
    rng = np.random.default_rng(seed + 1)
    dy32 = rng.standard_normal((b, L, H, P)).astype(np.float32)
    dy_host = _bf16_bits(dy32) if dtype == "bf16" else dy32
    dfin = rng.standard_normal((b, H, P, N)).astype(np.float32) if with_dfinal else None
    t = to_device(inp)
    if dtype == "bf16":
        dy = torch.from_numpy(dy_host.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        dy = torch.from_numpy(dy_host).cuda()
    g = ssd.bwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], dy, chunk=chunk, init_state=t["init"],
                dfinal=None if dfin is None else torch.from_numpy(dfin).cuda())
    torch.cuda.synchronize()
    dy_ref = synth.bf16_bits_to_f32(dy_host) if dtype == "bf16" else dy32
    ref = recurrence_bwd_np(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, dy_ref, dfin)
    tol = tol or (1e-4 if dtype == "f32" else 2e-2)
    tol_sc = tol_sc or (1e-4 if dtype == "f32" else 2e-2)
    errs = {}
    for name in ("dx", "dB", "dC", "dD", "ddt", "dA") + (("dinit",) if init else ()):
        got = g[name].float().cpu().numpy()
        errs[name] = rel(got, ref[name])
    for name, err in errs.items():
        bound = tol_sc if name in ("ddt", "dA") else tol
        assert err <= bound, (name, err, errs)
    return errs


def test_f32_small_groups_ragged():
    run_case("f32", 2, 100, 4, 16, 8, 2, 64, seed=3)


def test_f32_many_sequences_unit_scale_cumsum():
    # 64 sequences x 10 chunks of 64 tokens x 8 heads = 640 tiles: the adjoint scan's unit-scale
    # chunk_cumsum runs in the persistent TMA kernel (runs of 2 tokens per lane).  Short
    # sequences: float32 dA loses accuracy with sequence length (its two terms cancel), which
    # this test is not about.
    run_case("f32", 64, 617, 8, 16, 16, 1, 64, seed=23)


def test_f32_no_init_no_dfinal():
    run_case("f32", 1, 70, 2, 16, 16, 1, 64, init=False, with_dfinal=False, seed=5)


@pytest.mark.parametrize("G", [1, 2])
def test_bf16_tensor_core_shapes(G):
    # P = 64, N = 128, chunk 256: the forward-again and adjoint scans in float32 (CUDA cores),
    # the role-swapped scans as head-dim-64 scans on the tensor cores; 600 tokens: ragged end
    run_case("bf16", 2, 600, 4, 64, 128, G, 256, seed=7 + G)


def test_bf16_state_64_all_tensor_core():
    # N = 64: the role-swapped scans have head dim 64 and state 64, tensor-core shapes too
    run_case("bf16", 1, 512, 4, 64, 64, 1, 256, seed=11)


@pytest.mark.slow
def test_bf16_mamba2_130m_layer_full():
    # the 130M layer as the bench times it (b4 L2048 H24 P64 N128 G1, chunk 256, no init), every
    # gradient against the float64 adjoint over the whole tensor
    errs = run_case("bf16", 4, 2048, 24, 64, 128, 1, 256, init=False, seed=19)
    assert max(errs.values()) > 0.0

