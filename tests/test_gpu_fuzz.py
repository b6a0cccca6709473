"""Seeded random shapes through the forward and backward passes, against the float64 oracles.

The named workloads and edge cases (test_gpu_parity.py, test_gpu_bwd.py) pin chosen shapes;
these cases draw the shape itself -- batch, length (ragged or not), heads, groups, head dim,
state size, chunk, I/O dtype, with or without an initial state and D -- from a fixed seed, so
that each run covers the same mix of tensor-core and CUDA-core paths (P = 64 with chunk 128 or
256 and N in {64, 128} or a wide state take the tensor cores for bf16; the rest run on the CUDA
cores) and any failure reproduces.  Head dims and state sizes are multiples of 8.  Bounds are
the forward's: 1e-4 of max|ref| for float32 I/O, 2e-2 for bf16 (y and final_state alike, and
every gradient), except dA: the backward forms it from dL/dcs_t = <dy_t, y_t - D x_t> -
dt_t <x_t, g_t B_t>, a difference of two float32 scan outputs that can cancel to a small
fraction of either, so its bound also admits 8 float32 roundings of the cancelling magnitudes,
S_h = sum_t dt_t sum_{s >= t} (|first term| + |second term|) (+ |<dfinal, final>| at the last
token), both terms taken in float64 from the oracles.  A dropped term or a wrong sign moves dA by
about |dA|, far above that on these cases.
"""
import numpy as np
import pytest

from oracle.ref_bwd import recurrence_bwd_np
from state_space_model_02_gb300 import ssd, synth

from util import TOL, gather_y, oracle_pairs, rel, to_device, y_to_numpy

EPS32 = 2.0 ** -24

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _forward_cases(n=24, seed=20241203):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        chunk = int(rng.choice([64, 128, 256]))
        bf16 = bool(rng.random() < 0.6)
        # half the bf16 cases take the tensor-core shapes (P = 64, N in {64, 128} or wide)
        if bf16 and rng.random() < 0.5:
            P = 64
            chunk = int(rng.choice([128, 256]))
            N = int(rng.choice([64, 128, 256 if chunk == 256 else 192]))
        else:
            P = int(rng.choice([16, 32, 48, 64, 80, 96, 128]))
            N = int(rng.choice([16, 32, 48, 64, 96, 128, 192]))
        H = int(rng.integers(1, 9))
        G = int(rng.choice([g for g in (1, 2, 3, 4) if H % g == 0]))
        L = int(rng.integers(1, 700))
        b = int(rng.integers(1, 3))
        cases.append(dict(batch=b, seqlen=L, nheads=H, headdim=P, dstate=N, ngroups=G, chunk=chunk,
                          io_dtype="bf16" if bf16 else "f32", init=bool(rng.random() < 0.5),
                          with_D=bool(rng.random() < 0.8), seed=1000 + i))
    return cases


FORWARD = _forward_cases()


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_02_gb300 import build as cuda_build

    cuda_build.build()
    ssd.load_library()


@pytest.mark.parametrize("case", FORWARD, ids=["f%02d" % i for i in range(len(FORWARD))])
def test_forward_random_shape(case):
    inp = synth.make_inputs(**case)
    t = to_device(inp)
    y, fin = ssd.fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], chunk=inp.chunk, init_state=t["init"])
    torch.cuda.synchronize()
    y, fin = y_to_numpy(y), fin.cpu().numpy()
    b, L, H, P = inp.x.shape
    pairs = [(bb, hh) for bb in range(b) for hh in range(H)]
    out = oracle_pairs(inp, pairs)
    tol = TOL[inp.io_dtype]
    ey = rel(gather_y(y, pairs), out["y"])
    ef = rel(np.stack([fin[bb, hh] for bb, hh in pairs]), out["final"])
    assert ey <= tol and ef <= tol, "y err %.3e, final err %.3e (tol %.0e) for %s" % (ey, ef, tol, case)


def _backward_cases(n=8, seed=20241204):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        bf16 = bool(rng.random() < 0.5)
        P = 64 if (bf16 and rng.random() < 0.5) else int(rng.choice([16, 32, 64]))
        N = int(rng.choice([16, 32, 64, 128]))
        H = int(rng.integers(1, 5))
        G = int(rng.choice([g for g in (1, 2) if H % g == 0]))
        # short sequences: float32 dA loses accuracy with length (its two terms cancel)
        cases.append(dict(b=int(rng.integers(1, 3)), L=int(rng.integers(1, 300)), H=H, P=P, N=N, G=G,
                          chunk=int(rng.choice([64, 128, 256])), dtype="bf16" if bf16 else "f32",
                          init=bool(rng.random() < 0.5), dfinal=bool(rng.random() < 0.5), seed=2000 + i))
    return cases


BACKWARD = _backward_cases()


def da_bound(inp, dy_ref, dfin, ref, tol):
    """dA's bound: tol x max|dA|, or 8 float32 roundings of the magnitudes its terms cancel from."""
    b, L, H, P = inp.x.shape
    pairs = [(bb, hh) for bb in range(b) for hh in range(H)]
    fwd = oracle_pairs(inp, pairs)
    y = np.zeros((b, L, H, P))
    fin = np.zeros((b, H, P, inp.B.shape[3]))
    for k, (bb, hh) in enumerate(pairs):
        y[bb, :, hh] = fwd["y"][k]
        fin[bb, hh] = fwd["final"][k]
    x = synth.bf16_bits_to_f32(inp.x) if inp.io_dtype == "bf16" else inp.x
    x = np.asarray(x, np.float64)
    dt = inp.dt.astype(np.float64)
    Dv = (np.zeros(H) if inp.D is None else inp.D.astype(np.float64))[None, None, :, None]
    dy64 = np.asarray(dy_ref, np.float64)
    mag = np.abs(np.einsum("blhp,blhp->blh", dy64, y - Dv * x)) + \
        np.abs(np.einsum("blhp,blhp->blh", x, ref["dx"] - Dv * dy64))
    if dfin is not None:
        mag[:, -1] += np.abs(np.einsum("bhpn,bhpn->bh", np.asarray(dfin, np.float64), fin))
    S = np.einsum("blh,blh->h", dt, np.cumsum(mag[:, ::-1], axis=1)[:, ::-1]).max()
    return max(tol * np.abs(ref["dA"]).max(), 8 * EPS32 * S), S


@pytest.mark.parametrize("case", BACKWARD, ids=["b%02d" % i for i in range(len(BACKWARD))])
def test_backward_random_shape(case):
    c = case
    inp = synth.make_inputs(c["b"], c["L"], c["H"], c["P"], c["N"], c["G"], chunk=c["chunk"], io_dtype=c["dtype"],
                            init=c["init"], seed=c["seed"])
    rng = np.random.default_rng(c["seed"] + 1)
    dy32 = rng.standard_normal((c["b"], c["L"], c["H"], c["P"])).astype(np.float32)
    dfin = rng.standard_normal((c["b"], c["H"], c["P"], c["N"])).astype(np.float32) if c["dfinal"] else None
    t = to_device(inp)
    if c["dtype"] == "bf16":
        dy_bits = synth.to_bf16_bits(dy32)
        dy = torch.from_numpy(dy_bits.view(np.int16)).view(torch.bfloat16).cuda()
        dy_ref = synth.bf16_bits_to_f32(dy_bits)
    else:
        dy = torch.from_numpy(dy32).cuda()
        dy_ref = dy32
    g = ssd.bwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], dy, chunk=c["chunk"], init_state=t["init"],
                dfinal=None if dfin is None else torch.from_numpy(dfin).cuda())
    torch.cuda.synchronize()
    ref = recurrence_bwd_np(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, dy_ref, dfin)
    tol = TOL[c["dtype"]]
    names = ("dx", "dB", "dC", "dD", "ddt") + (("dinit",) if c["init"] else ())
    errs = {n: rel(g[n].float().cpu().numpy(), ref[n]) for n in names}
    bad = {n: e for n, e in errs.items() if e > tol}
    assert not bad, "errors above %.0e: %s for %s" % (tol, bad, case)
    got_dA = g["dA"].float().cpu().numpy()
    err = np.abs(got_dA - ref["dA"]).max()
    bound, S = da_bound(inp, dy_ref, dfin, ref, tol)
    assert err <= bound, "dA err %.3e above %.3e (|dA| %.3e, S %.3e) for %s" % (
        err, bound, np.abs(ref["dA"]).max(), S, case)
