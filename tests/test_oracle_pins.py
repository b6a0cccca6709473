"""Pins of the float64 oracle against things other than itself (CPU only).

Each test ties an oracle function to a hand-worked example, a closed form, a
library routine, brute force, or an invariant that the mathematics fixes, so a
dropped term, wrong sign or index, or transposed operand in the oracle fails at
least one of them.  The mutation tests at the end plant such mistakes in a
copy of the oracle and check that the pins notice.
"""
import math
import os

import numpy as np
import pytest

from oracle import ref
from state_space_model_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = np.array([float(v) for v in rest])
    return vals


def _rand(b, L, H, P, N, G=1, dtype="f32", init=True, seed=1, a_range=(1.0, 16.0), chunk=64):
    return synth.make_inputs(b, L, H, P, N, G, chunk=chunk, io_dtype=dtype, init=init, seed=seed,
                             a_range=a_range)


def _run(inp, **kw):
    return ref.recurrence(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, chunk=inp.chunk, **kw)


def _to_bhlp(y, b, H):
    # oracle y is (nsel, L, P) over pairs (b, h) in row-major order
    nsel, L, P = y.shape
    return y.reshape(b, H, L, P).transpose(0, 2, 1, 3)


# --------------------------------------------------------------------------- golden


def test_golden_scalar_recurrence():
    g = _load_golden("scalar_halving_decay.txt")
    L = int(g["L"][0])
    x = g["x"].astype(np.float32).reshape(1, L, 1, 1)
    B = g["B"].astype(np.float32).reshape(1, L, 1, 1)
    C = g["C"].astype(np.float32).reshape(1, L, 1, 1)
    dt = g["dt"].astype(np.float32).reshape(1, L, 1)
    A = g["A"].astype(np.float32)
    D = g["D"].astype(np.float32)
    init = g["init"].astype(np.float32).reshape(1, 1, 1, 1)
    Q = int(g["chunk"][0])
    out = ref.recurrence(x, dt, A, B, C, D, init, chunk=Q, want_chunk_in=True)
    np.testing.assert_allclose(out["y"].ravel(), g["y"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(out["final"].ravel(), g["final"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(out["chunk_in"].ravel(), g["chunk_in"], rtol=1e-6, atol=1e-6)
    S = ref.chunk_states(x, dt, A, B, Q)
    np.testing.assert_allclose(S.ravel(), g["chunk_states"], rtol=1e-6, atol=1e-6)
    cs2, dtT = ref.cumsum_log2(dt, A, Q)
    np.testing.assert_allclose(cs2.ravel(), g["cs2"], rtol=1e-6, atol=1e-6)
    np.testing.assert_array_equal(dtT.ravel(), g["dt"])
    # the NumPy forms reproduce the same hand-worked numbers
    yq, fq = ref.quadratic(x, dt, A, B, C, D, init)
    np.testing.assert_allclose(yq.ravel(), g["y"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(fq.ravel(), g["final"], rtol=1e-6, atol=1e-6)
    yc, fc, cin, Sc = ref.chunked(x, dt, A, B, C, D, init, chunk=Q)
    np.testing.assert_allclose(yc.ravel(), g["y"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(cin.ravel(), g["chunk_in"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(Sc.ravel(), g["chunk_states"], rtol=1e-6, atol=1e-6)


# ----------------------------------------------------------------- brute force / dual form


@pytest.mark.parametrize("shape", [
    dict(b=1, L=37, H=2, P=3, N=5, G=1),
    dict(b=2, L=64, H=4, P=4, N=8, G=2),
    dict(b=1, L=128, H=3, P=8, N=4, G=3),
])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_recurrence_matches_quadratic_dual_form(shape, dtype):
    inp = _rand(shape["b"], shape["L"], shape["H"], shape["P"], shape["N"], shape["G"], dtype=dtype,
                a_range=(0.05, 4.0))
    out = _run(inp)
    yq, fq = ref.quadratic(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init)
    y = _to_bhlp(out["y"], shape["b"], shape["H"])
    assert ref.rel_err(y, yq) < 1e-12
    assert ref.rel_err(out["final"].reshape(fq.shape), fq) < 1e-12


def test_c_recurrence_matches_numpy_twin():
    inp = _rand(2, 50, 4, 3, 6, 2, dtype="bf16")
    out = _run(inp)
    yn, fn = ref.recurrence_np(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init)
    assert ref.rel_err(_to_bhlp(out["y"], 2, 4), yn) < 1e-13
    assert ref.rel_err(out["final"].reshape(fn.shape), fn) < 1e-13


# ------------------------------------------------------------- chunked form, chunk invariance


@pytest.mark.parametrize("Q", [16, 32, 64, 256])
@pytest.mark.parametrize("L", [200, 256])
def test_chunked_form_matches_recurrence(Q, L):
    inp = _rand(1, L, 2, 4, 8, 1, dtype="bf16", a_range=(0.01, 2.0), chunk=Q)
    out = _run(inp, want_chunk_in=True)
    yc, fc, cin, S = ref.chunked(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, chunk=Q)
    assert ref.rel_err(_to_bhlp(out["y"], 1, 2), yc) < 1e-12
    assert ref.rel_err(out["final"].reshape(fc.shape), fc) < 1e-12
    # state entering each chunk: oracle (nsel, nc, P, N) vs chunked (b, nc, H, P, N)
    assert ref.rel_err(out["chunk_in"], cin[0].transpose(1, 0, 2, 3)) < 1e-12
    Sc = ref.chunk_states(inp.x, inp.dt, inp.A, inp.B, Q)
    assert ref.rel_err(Sc, S[0].transpose(1, 0, 2, 3)) < 1e-12


def test_chunk_states_chain_to_chunk_inputs():
    # linearity across a chunk: h_in[c+1] = exp(sum_c dt*A) h_in[c] + S[c]
    Q = 32
    inp = _rand(1, 160, 3, 4, 5, 1, dtype="f32", a_range=(0.02, 1.0), chunk=Q)
    out = _run(inp, want_chunk_in=True)
    S = ref.chunk_states(inp.x, inp.dt, inp.A, inp.B, Q)
    dt = inp.dt.astype(np.float64)
    for s, h in enumerate(range(3)):
        for c in range(4):
            tot = math.exp(float(np.sum(dt[0, c * Q:(c + 1) * Q, h]) * float(inp.A[h])))
            nxt = tot * out["chunk_in"][s, c] + S[s, c]
            assert ref.rel_err(nxt, out["chunk_in"][s, c + 1]) < 1e-12


# ------------------------------------------------------------------------- closed forms


def test_zero_decay_is_causal_prefix_sum():
    # A = 0 and dt = delta: h_t = delta * sum_{s<=t} x_s (x) B_s, y_t = h_t . C_t (+ D x_t)
    b, L, H, P, N = 1, 90, 2, 3, 4
    inp = _rand(b, L, H, P, N, dtype="f32", init=False)
    delta = np.float32(0.0625)
    inp.A[:] = 0.0
    inp.dt[:] = delta
    out = _run(inp)
    x = inp.x.astype(np.float64)
    Bm = inp.B.astype(np.float64)[:, :, 0]
    Cm = inp.C.astype(np.float64)[:, :, 0]
    outer = x[..., :, None] * Bm[:, :, None, None, :]           # (b, L, H, P, N)
    states = float(delta) * np.cumsum(outer, axis=1)
    y = np.einsum("blhpn,bln->blhp", states, Cm) + inp.D.astype(np.float64)[None, None, :, None] * x
    assert ref.rel_err(_to_bhlp(out["y"], b, H), y) < 1e-12
    assert ref.rel_err(out["final"].reshape(b, H, P, N), states[:, -1]) < 1e-12


def test_final_state_explicit_unroll():
    # final = sum_t exp(sum_{s>t} dt_s A) dt_t x_t (x) B_t + exp(sum_s dt_s A) h0
    b, L, H, P, N = 1, 70, 2, 3, 4
    inp = _rand(b, L, H, P, N, dtype="f32", a_range=(0.05, 1.0))
    out = _run(inp, want_y=False)
    dt, A = inp.dt.astype(np.float64), inp.A.astype(np.float64)
    x, Bm = inp.x.astype(np.float64), inp.B.astype(np.float64)[:, :, 0]
    for h in range(H):
        acc = np.zeros((P, N))
        for t in range(L):
            later = sum(float(dt[0, s, h]) for s in range(t + 1, L))
            acc += math.exp(later * A[h]) * dt[0, t, h] * np.outer(x[0, t, h], Bm[0, t])
        acc += math.exp(float(np.sum(dt[0, :, h])) * A[h]) * inp.init[0, h].astype(np.float64)
        assert ref.rel_err(out["final"][h], acc) < 1e-12


@pytest.mark.parametrize("split", [64, 100])   # aligned and not aligned to the chunk
def test_split_and_resume_matches_unsplit(split):
    b, L, H, P, N, Q = 2, 256, 3, 4, 6, 64
    inp = _rand(b, L, H, P, N, dtype="bf16", chunk=Q, a_range=(0.01, 2.0))
    full = _run(inp)
    a = ref.recurrence(inp.x[:, :split], inp.dt[:, :split], inp.A, inp.B[:, :split],
                       inp.C[:, :split], inp.D, inp.init, chunk=Q)
    mid = a["final"].reshape(b, H, P, N).astype(np.float32)
    # the resumed half starts from the float64 state rounded to float32 (the
    # init-state I/O dtype), so compare at float32 resolution
    bpart = ref.recurrence(inp.x[:, split:], inp.dt[:, split:], inp.A, inp.B[:, split:],
                           inp.C[:, split:], inp.D, mid, chunk=Q)
    y = np.concatenate([_to_bhlp(a["y"], b, H), _to_bhlp(bpart["y"], b, H)], axis=1)
    assert ref.rel_err(y, _to_bhlp(full["y"], b, H)) < 1e-6
    assert ref.rel_err(bpart["final"], full["final"]) < 1e-6


def test_single_token_closed_form():
    # L = 1: y = dt (C.B) x + exp(dt A) (C . h0) + D x ; final = exp(dt A) h0 + dt x (x) B
    inp = _rand(1, 1, 3, 4, 5, dtype="f32")
    out = _run(inp)
    dt, A, D = inp.dt[0, 0].astype(np.float64), inp.A.astype(np.float64), inp.D.astype(np.float64)
    x, Bv, Cv = inp.x[0, 0].astype(np.float64), inp.B[0, 0, 0].astype(np.float64), inp.C[0, 0, 0].astype(np.float64)
    h0 = inp.init[0].astype(np.float64)
    for h in range(3):
        y = dt[h] * (Cv @ Bv) * x[h] + math.exp(dt[h] * A[h]) * (h0[h] @ Cv) + D[h] * x[h]
        fin = math.exp(dt[h] * A[h]) * h0[h] + dt[h] * np.outer(x[h], Bv)
        assert ref.rel_err(out["y"][h, 0], y) < 1e-14
        assert ref.rel_err(out["final"][h], fin) < 1e-14


def test_scalar_case_is_first_order_linear_filter():
    # P = N = H = 1, constant dt: h_t = a h_{t-1} + u_t is an IIR filter 1 / (1 - a z^-1)
    signal = pytest.importorskip("scipy.signal")
    L = 300
    inp = _rand(1, L, 1, 1, 1, dtype="f32", init=False, a_range=(0.5, 3.0))
    inp.dt[:] = np.float32(0.05)
    out = _run(inp)
    a = math.exp(float(inp.dt[0, 0, 0]) * float(inp.A[0]))
    u = float(inp.dt[0, 0, 0]) * inp.x[0, :, 0, 0].astype(np.float64) * inp.B[0, :, 0, 0].astype(np.float64)
    h = signal.lfilter([1.0], [1.0, -a], u)
    y = h * inp.C[0, :, 0, 0].astype(np.float64) + float(inp.D[0]) * inp.x[0, :, 0, 0].astype(np.float64)
    assert ref.rel_err(out["y"][0, :, 0], y) < 1e-12
    assert abs(out["final"][0, 0, 0] - h[-1]) <= 1e-12 * max(1.0, abs(h[-1]))


def test_linearity_in_x_and_init():
    inp = _rand(1, 80, 2, 3, 4, dtype="f32", init=True)
    base = _run(inp)
    inp2 = synth.SSDInputs(x=inp.x * 2, dt=inp.dt, A=inp.A, B=inp.B, C=inp.C, D=inp.D,
                           init=inp.init * 2, chunk=inp.chunk, io_dtype="f32")
    dbl = _run(inp2)
    assert ref.rel_err(dbl["y"], 2 * base["y"]) < 1e-14
    assert ref.rel_err(dbl["final"], 2 * base["final"]) < 1e-14


def test_cumsum_log2_is_log_of_decay_product():
    # exp2(cs2[i]) must equal the product of per-token decays exp(dt_s A) over s <= i in the
    # chunk; positions past the sequence end carry dt = 0 and leave cs2 unchanged.
    Q = 64
    inp = _rand(2, 150, 3, 1, 1, dtype="f32", chunk=Q)
    cs2, dtT = ref.cumsum_log2(inp.dt, inp.A, Q)
    dt, A = inp.dt.astype(np.float64), inp.A.astype(np.float64)
    for b in range(2):
        for h in range(3):
            for c in range(3):
                prod = 1.0
                for i in range(Q):
                    t = c * Q + i
                    if t < 150:
                        prod *= math.exp(dt[b, t, h] * A[h])
                        assert dtT[b, h, c, i] == inp.dt[b, t, h]
                    else:
                        assert dtT[b, h, c, i] == 0.0
                    assert abs(2.0 ** cs2[b, h, c, i] - prod) <= 1e-12 * prod


# ------------------------------------------------------------------- input generator


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    a = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10,
                        np.array([1.00390625, 1.01171875, -2.5, 0.0, 3.0e-39], np.float32)])
    ours = synth.to_bf16_bits(a)
    theirs = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, theirs)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(ours),
                                  torch.from_numpy(a).to(torch.bfloat16).float().numpy())


def test_generator_is_deterministic_and_in_range():
    a = synth.make_config("tiny_fp32")
    b = synth.make_config("tiny_fp32")
    for k in ("x", "dt", "A", "B", "C", "D"):
        np.testing.assert_array_equal(getattr(a, k), getattr(b, k))
    assert a.dt.min() >= np.float32(1e-3) and a.dt.max() <= np.float32(0.1)
    assert np.all(a.A <= -1.0) and np.all(a.A >= -16.0)
    assert a.init is None


def test_generator_distribution_matches_recipe():
    # dt = clip(softplus(N(-3, 1)), 1e-3, 0.1): the clipped fractions are normal tail masses;
    # A = -exp(U(0, ln 16)); x ~ N(0, 1), rounded to bf16
    import math
    inp = synth.make_inputs(batch=1, seqlen=2048, nheads=2048, headdim=2, dstate=2, chunk=256,
                            io_dtype="bf16", seed=23)
    dt = inp.dt.ravel()
    n = dt.size

    def tail_above(v):  # P(N(-3, 1) > v)
        return 0.5 * math.erfc((v + 3.0) / math.sqrt(2.0))

    p_hi = tail_above(math.log(math.expm1(0.1)))           # about 0.227
    p_lo = 1.0 - tail_above(math.log(math.expm1(1e-3)))    # about 5e-5
    f_hi = np.mean(dt == np.float32(0.1))
    f_lo = np.mean(dt == np.float32(1e-3))
    assert abs(f_hi - p_hi) < 5 * math.sqrt(p_hi * (1 - p_hi) / n)
    assert abs(f_lo - p_lo) < 5 * math.sqrt(p_lo * (1 - p_lo) / n) + 1.0 / n
    u = np.log(-inp.A.astype(np.float64)) / math.log(16.0)   # U(0, 1)
    assert abs(u.mean() - 0.5) < 5 * math.sqrt(1.0 / 12.0 / u.size)
    assert u.min() >= 0.0 and u.max() <= 1.0
    x = synth.bf16_bits_to_f32(inp.x).astype(np.float64).ravel()
    assert abs(x.mean()) < 5.0 / math.sqrt(x.size) and abs(x.std() - 1.0) < 0.01


# ------------------------------------------------------------------------ mutations


def _mutant_recurrence(x, dt, A, B, C, D, init, mistake):
    """Copy of the NumPy recurrence with one planted mistake (CPU only)."""
    x, B, C = ref.widen(x), ref.widen(B), ref.widen(C)
    dt, A = np.asarray(dt, np.float64), np.asarray(A, np.float64)
    b, L, H, P = x.shape
    N = B.shape[3]
    h = np.asarray(init, np.float64).copy()
    y = np.empty((b, L, H, P))
    sign = -1.0 if mistake == "sign" else 1.0
    for t in range(L):
        Bt, Ct = B[:, t, [0] * H], C[:, t, [0] * H]
        if mistake == "transpose":
            Bt, Ct = Ct, Bt
        decay = np.exp(sign * dt[:, t] * A)
        hn = decay[..., None, None] * h + (dt[:, t][..., None] * x[:, t])[..., None] * Bt[:, :, None, :]
        read = h if mistake == "exclusive" else hn
        y[:, t] = np.einsum("bhpn,bhn->bhp", read, Ct)
        if mistake != "drop_D":
            y[:, t] += np.asarray(D, np.float64)[:, None] * x[:, t]
        h = hn
    return y, h


@pytest.mark.parametrize("mistake", ["sign", "transpose", "exclusive", "drop_D"])
def test_pins_catch_planted_mistakes(mistake):
    inp = _rand(1, 48, 2, 3, 4, dtype="f32", a_range=(0.5, 4.0))
    yq, fq = ref.quadratic(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init)
    ym, fm = _mutant_recurrence(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, mistake)
    assert max(ref.rel_err(ym, yq), ref.rel_err(fm, fq)) > 1e-3
    # and the unmutated copy passes the same pin
    y0, f0 = _mutant_recurrence(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, None)
    assert ref.rel_err(y0, yq) < 1e-12 and ref.rel_err(f0, fq) < 1e-12
