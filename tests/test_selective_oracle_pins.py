"""Pins of the float64 Mamba-1 selective-scan oracle against things other than itself (CPU).

Source of the definition: "3.3 Hardware-aware algorithm and GPU memory hierarchy"
(booiljung.github.io), section 2.1 (zero-order hold), section 3 (the fused steps: load,
discretise, scan, multiply by C) and section 4.1 (first-order linear recurrence, associative).
Each pin ties the oracle to a hand-worked example, a library routine (scipy's lfilter and
ODE integrator), a closed form or an invariant; the mutation tests plant mistakes in a copy
of the oracle's NumPy twin and check that the pins catch them.
"""
import math
import os

import numpy as np
import pytest

from oracle import selective as sel
from oracle.ref import widen
from state_space_model_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *rest = line.split()
                vals[k] = np.array([float(v) for v in rest])
    return vals


def _c_oracle(x, delta, A, B, C, Dskip=None, init=None):
    o = sel.selective_scan(x, delta, A, B, C, Dskip, init)
    return o["y"], o["final"]


IMPLS = {"c": _c_oracle, "numpy": sel.selective_scan_np}


def _f32(*arrays):
    return [None if a is None else np.ascontiguousarray(a, np.float32) for a in arrays]


# ---------------------------------------------------------------------------- the pins


def pin_golden(impl):
    g = _golden("selective_one_state.txt")
    L = int(g["L"][0])
    x, d, B, C = _f32(g["x"].reshape(1, L, 1), g["delta"].reshape(1, L, 1), g["B"].reshape(1, L, 1),
                      g["C"].reshape(1, L, 1))
    A, Dk, h0 = _f32(g["A"].reshape(1, 1), g["Dskip"], g["init"].reshape(1, 1, 1))
    y, fin = impl(x, d, A, B, C, Dk, h0)
    # float32 rounding of A = -ln 2 moves the values by ~1e-7 relative
    return np.allclose(y.ravel(), g["y"], rtol=1e-6, atol=1e-6) and \
        np.allclose(fin.ravel(), g["final"], rtol=1e-6, atol=1e-6)


def pin_lfilter(impl):
    # constant delta and A: a first-order IIR filter of u_t = B_t x_t, read out by C_t
    from scipy.signal import lfilter
    rng = np.random.default_rng(5)
    L, dv, a = 300, 0.05, -3.0
    x, B, C = (rng.standard_normal((1, L, 1)).astype(np.float32) for _ in range(3))
    d = np.full((1, L, 1), dv, np.float32)
    A = np.array([[a]], np.float32)
    y, fin = impl(x, d, A, B, C)
    af, dvf = float(np.float32(a)), float(np.float32(dv))
    abar = math.exp(dvf * af)
    gain = math.expm1(dvf * af) / af
    h = lfilter([gain], [1.0, -abar], widen(B).ravel() * widen(x).ravel())
    return np.allclose(y.ravel(), widen(C).ravel() * h, rtol=1e-10, atol=1e-12) and \
        abs(fin.ravel()[0] - h[-1]) < 1e-12


def pin_zoh_is_exact_for_piecewise_constant_input(impl):
    # The zero-order hold is the exact solution of h' = A h + B x over a step of length delta
    # with x and B held constant: integrate that ODE numerically and compare the states.
    from scipy.integrate import solve_ivp
    rng = np.random.default_rng(7)
    L, N = 12, 3
    x = rng.standard_normal((1, L, 1)).astype(np.float32)
    B = rng.standard_normal((1, L, N)).astype(np.float32)
    C = rng.standard_normal((1, L, N)).astype(np.float32)
    d = rng.uniform(0.05, 0.6, size=(1, L, 1)).astype(np.float32)
    A = np.array([[-0.5, -2.0, -7.0]], np.float32)
    h0 = rng.standard_normal((1, 1, N)).astype(np.float32)
    y, fin = impl(x, d, A, B, C, None, h0)
    Ad = A.astype(np.float64).ravel()
    h = h0.astype(np.float64).ravel()
    ys = []
    for t in range(L):
        u = B[0, t].astype(np.float64) * float(x[0, t, 0])
        sol = solve_ivp(lambda _, s: Ad * s + u, (0.0, float(d[0, t, 0])), h, rtol=1e-12, atol=1e-14,
                        method="DOP853")
        h = sol.y[:, -1]
        ys.append(float(C[0, t].astype(np.float64) @ h))
    return np.allclose(y.ravel(), ys, rtol=1e-8, atol=1e-10) and np.allclose(fin.ravel(), h, rtol=1e-8,
                                                                              atol=1e-10)


def pin_zero_A_is_a_prefix_sum(impl):
    # A = 0: Abar = 1 and Bbar = delta B (the limit), so h_t = h_0 + sum_{s<=t} delta_s B_s x_s
    rng = np.random.default_rng(9)
    b, L, D, N = 2, 20, 3, 4
    x = rng.standard_normal((b, L, D)).astype(np.float32)
    d = rng.uniform(0.01, 0.1, (b, L, D)).astype(np.float32)
    B, C = (rng.standard_normal((b, L, N)).astype(np.float32) for _ in range(2))
    A = np.zeros((D, N), np.float32)
    h0 = rng.standard_normal((b, D, N)).astype(np.float32)
    y, fin = impl(x, d, A, B, C, None, h0)
    inc = d.astype(np.float64)[..., None] * x.astype(np.float64)[..., None] * B.astype(np.float64)[:, :, None, :]
    h = h0.astype(np.float64)[:, None] + np.cumsum(inc, axis=1)              # (b, L, D, N)
    y_ref = np.einsum("bldn,bln->bld", h, C.astype(np.float64))
    return np.allclose(y, y_ref, rtol=1e-11, atol=1e-11) and np.allclose(fin, h[:, -1], rtol=1e-11, atol=1e-11)


def pin_associative_scan(impl):
    # Section 4.1: (a, b) pairs combine associatively; a Hillis-Steele inclusive scan of
    # (Abar_t, Bbar_t x_t) must give the same states as the token loop.
    inp = synth.make_selective_inputs(1, 64, 5, 6, io_dtype="f32", init=True, seed=11)
    y, fin = impl(inp.x, inp.delta, inp.A, inp.B, inp.C, None, inp.init)
    dl, x, B, C = (widen(a)[0] for a in (inp.delta, inp.x, inp.B, inp.C))
    A = inp.A.astype(np.float64)
    w = dl[:, :, None] * A[None]                                   # (L, D, N)
    a = np.exp(w)
    bb = np.expm1(w) / A[None] * B[:, None, :] * x[:, :, None]
    a, bb = a.copy(), bb.copy()
    step = 1
    while step < a.shape[0]:
        a_prev, b_prev = a[:-step].copy(), bb[:-step].copy()
        bb[step:] = a[step:] * b_prev + bb[step:]
        a[step:] = a[step:] * a_prev
        step *= 2
    h = a * inp.init.astype(np.float64)[0][None] + bb               # states after every token
    y_ref = np.einsum("ldn,ln->ld", h, C)
    return np.allclose(y[0], y_ref, rtol=1e-10, atol=1e-10) and np.allclose(fin[0], h[-1], rtol=1e-10,
                                                                             atol=1e-10)


def pin_split_resume(impl):
    inp = synth.make_selective_inputs(2, 50, 7, 8, io_dtype="f32", init=True, seed=13)
    y, fin = impl(inp.x, inp.delta, inp.A, inp.B, inp.C, inp.D, inp.init)
    k = 23
    sl = lambda a, s: np.ascontiguousarray(a[:, s])
    y1, f1 = impl(sl(inp.x, slice(0, k)), sl(inp.delta, slice(0, k)), inp.A, sl(inp.B, slice(0, k)),
                  sl(inp.C, slice(0, k)), inp.D, inp.init)
    y2, f2 = impl(sl(inp.x, slice(k, None)), sl(inp.delta, slice(k, None)), inp.A, sl(inp.B, slice(k, None)),
                  sl(inp.C, slice(k, None)), inp.D, f1.astype(np.float32))
    # the resumed half starts from the float32-rounded state, hence the looser bound there
    return np.allclose(y[:, :k], y1, rtol=1e-13, atol=1e-13) and np.allclose(y[:, k:], y2, rtol=1e-5, atol=1e-6) \
        and np.allclose(fin, f2, rtol=1e-5, atol=1e-6)


def pin_skip_and_linearity(impl):
    # y is linear in (x, init) jointly; the skip adds Dskip x exactly
    inp = synth.make_selective_inputs(1, 30, 4, 5, io_dtype="f32", init=True, seed=17)
    y0, _ = impl(inp.x, inp.delta, inp.A, inp.B, inp.C, None, inp.init)
    y1, _ = impl(inp.x, inp.delta, inp.A, inp.B, inp.C, inp.D, inp.init)
    y2, _ = impl((2 * inp.x).astype(np.float32), inp.delta, inp.A, inp.B, inp.C, None,
                 (2 * inp.init).astype(np.float32))
    skip = inp.D.astype(np.float64)[None, None] * inp.x.astype(np.float64)
    return np.allclose(y1 - y0, skip, rtol=1e-12, atol=1e-12) and np.allclose(y2, 2 * y0, rtol=1e-12, atol=1e-12)


PINS = [pin_golden, pin_lfilter, pin_zoh_is_exact_for_piecewise_constant_input, pin_zero_A_is_a_prefix_sum,
        pin_associative_scan, pin_split_resume, pin_skip_and_linearity]


@pytest.mark.parametrize("impl", sorted(IMPLS))
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin, impl):
    assert pin(IMPLS[impl])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_c_oracle_matches_numpy_twin(dtype):
    inp = synth.make_selective_inputs(3, 41, 10, 16, io_dtype=dtype, init=True, seed=19)
    yc, fc = _c_oracle(inp.x, inp.delta, inp.A, inp.B, inp.C, inp.D, inp.init)
    yn, fn = sel.selective_scan_np(inp.x, inp.delta, inp.A, inp.B, inp.C, inp.D, inp.init)
    assert np.abs(yc - yn).max() <= 1e-12 * max(1.0, np.abs(yn).max())
    assert np.abs(fc - fn).max() <= 1e-12 * max(1.0, np.abs(fn).max())


# ------------------------------------------------------------- planted mistakes


def _mutant(kind):
    def impl(x, delta, A, B, C, Dskip=None, init=None):
        x, delta, B, C = (widen(a) for a in (x, delta, B, C))
        A = np.asarray(A, np.float64)
        b, L, D = x.shape
        N = B.shape[2]
        h = np.zeros((b, D, N)) if init is None else np.asarray(init, np.float64).copy()
        skip = np.zeros(D) if Dskip is None else np.asarray(Dskip, np.float64)
        y = np.empty((b, L, D))
        for t in range(L):
            w = delta[:, t, :, None] * A[None]
            safe = np.where(A == 0.0, 1.0, A)
            coef = np.where(A[None] == 0.0, delta[:, t, :, None], np.expm1(w) / safe[None])
            if kind == "euler_B":          # delta B instead of the zero-order hold
                coef = np.broadcast_to(delta[:, t, :, None], w.shape)
            Bt, Ct = B[:, t], C[:, t]
            if kind == "swap_BC":
                Bt, Ct = Ct, Bt
            h_old = h
            h = np.exp(w) * h + coef * Bt[:, None, :] * x[:, t, :, None]
            hy = h_old if kind == "exclusive" else h
            y[:, t] = np.einsum("bdn,bn->bd", hy, Ct) + (0 if kind == "no_skip" else skip * x[:, t])
            if kind == "decay_sign":
                h = h_old * np.exp(-w) + coef * Bt[:, None, :] * x[:, t, :, None]
        return y, h
    return impl


@pytest.mark.parametrize("kind", ["euler_B", "swap_BC", "exclusive", "no_skip", "decay_sign"])
def test_pins_catch_planted_mistakes(kind):
    impl = _mutant(kind)
    caught = []
    for pin in PINS:
        try:
            ok = pin(impl)
        except (FloatingPointError, ValueError, OverflowError):
            ok = False
        if not ok:
            caught.append(pin.__name__)
    assert caught, "no pin caught the planted mistake %r" % kind
