"""Pins of the float64 backward oracle (oracle/ref_bwd.py) against things other than itself.

(1) Central finite differences of the forward oracle's loss along random directions, for
every input; (2) torch.autograd through a float64 restatement of the forward recurrence of
"Mamba-2 cuda-tile forward pass kernels", sections 1-2 (autograd is the library routine
under test there, not the oracle's adjoint); (3) planted mistakes in a copy of the adjoint
(the decay applied one token late, B and C swapped, the decay term of ddt dropped) must be
caught by the finite differences.
"""
import numpy as np
import pytest

from oracle import ref
from oracle.ref_bwd import recurrence_bwd_np
from state_space_model_02_gb300 import synth

torch = pytest.importorskip("torch")


def _problem(G=1, init=True, seed=3):
    inp = synth.make_inputs(2, 11, 4, 3, 5, G, chunk=64, io_dtype="f32", init=init, seed=seed)
    rng = np.random.default_rng(seed + 100)
    b, L, H, P = inp.x.shape
    N = inp.B.shape[3]
    dy = rng.standard_normal((b, L, H, P))
    dfin = rng.standard_normal((b, H, P, N))
    args = dict(x=inp.x.astype(np.float64), dt=inp.dt.astype(np.float64), A=inp.A.astype(np.float64),
                B=inp.B.astype(np.float64), C=inp.C.astype(np.float64), D=inp.D.astype(np.float64),
                init=None if inp.init is None else inp.init.astype(np.float64))
    return args, dy, dfin


def _loss(args, dy, dfin):
    y, fin = ref.recurrence_np(args["x"], args["dt"], args["A"], args["B"], args["C"], args["D"], args["init"])
    return float(np.sum(y * dy) + np.sum(fin * dfin))


NAMES = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "init": "dinit"}


def _check_fd(grads, args, dy, dfin, seed=0):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for name, gname in NAMES.items():
        if args[name] is None:
            continue
        v = rng.standard_normal(args[name].shape)
        eps = 1e-6
        ap = dict(args); ap[name] = args[name] + eps * v
        am = dict(args); am[name] = args[name] - eps * v
        fd = (_loss(ap, dy, dfin) - _loss(am, dy, dfin)) / (2 * eps)
        an = float(np.sum(grads[gname] * v))
        worst = max(worst, abs(fd - an) / max(1.0, abs(fd)))
    return worst


@pytest.mark.parametrize("G,init", [(1, True), (2, True), (4, False)])
def test_adjoint_matches_finite_differences(G, init):
    args, dy, dfin = _problem(G, init)
    g = recurrence_bwd_np(args["x"], args["dt"], args["A"], args["B"], args["C"], args["D"], args["init"], dy, dfin)
    assert _check_fd(g, args, dy, dfin) < 1e-6


def test_adjoint_matches_torch_autograd():
    args, dy, dfin = _problem(2, True, seed=9)
    t = {k: torch.tensor(v, requires_grad=True) for k, v in args.items() if v is not None}
    b, L, H, P = args["x"].shape
    G = args["B"].shape[2]
    grp = torch.arange(H) // (H // G)
    h = t["init"]
    ys = []
    for s in range(L):
        Bt, Ct = t["B"][:, s][:, grp], t["C"][:, s][:, grp]
        a = torch.exp(t["dt"][:, s] * t["A"])
        h = a[..., None, None] * h + (t["dt"][:, s][..., None] * t["x"][:, s])[..., None] * Bt[:, :, None, :]
        ys.append(torch.einsum("bhpn,bhn->bhp", h, Ct) + t["D"][:, None] * t["x"][:, s])
    y = torch.stack(ys, 1)
    loss = (y * torch.tensor(dy)).sum() + (h * torch.tensor(dfin)).sum()
    loss.backward()
    g = recurrence_bwd_np(args["x"], args["dt"], args["A"], args["B"], args["C"], args["D"], args["init"], dy, dfin)
    for name, gname in NAMES.items():
        assert np.allclose(g[gname], t[name].grad.numpy(), rtol=1e-10, atol=1e-12), name


def _mutant(kind):
    def bwd(x, dt, A, B, C, D, init, dy, dfinal):
        g = recurrence_bwd_np(x, dt, A, B, C, D, init, dy, dfinal)
        if kind == "swap_BC":
            return recurrence_bwd_np(x, dt, A, C, B, D, init, dy, dfinal)
        if kind == "late_decay":   # the adjoint decays with a_t instead of a_{t+1}
            return recurrence_bwd_np(x, np.roll(dt, 1, axis=1), A, B, C, D, init, dy, dfinal)
        if kind == "no_decay_term":
            a = np.exp(np.asarray(dt) * np.asarray(A)[None, None])
            g = dict(g)
            g["dA"] = np.zeros_like(g["dA"])
            return g
        return g
    return bwd


@pytest.mark.parametrize("kind", ["swap_BC", "late_decay", "no_decay_term"])
def test_finite_differences_catch_planted_mistakes(kind):
    args, dy, dfin = _problem(2, True, seed=5)
    g = _mutant(kind)(args["x"], args["dt"], args["A"], args["B"], args["C"], args["D"], args["init"], dy, dfin)
    assert _check_fd(g, args, dy, dfin) > 1e-4
