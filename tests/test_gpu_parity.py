"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Metric: max|got - ref| / max|ref| over the compared tensor; bounds 1e-4 for float32 I/O and
2e-2 for bf16 I/O with float32 accumulation, for y and for final_state alike.  Small
problems are compared element by element in full; the full-size workloads on sampled
(batch, head) pairs, each of which the oracle recomputes over the whole sequence.
"""
import numpy as np
import pytest

from oracle import ref
from state_space_model_02_gb300 import ssd, synth

from util import TOL, gather_y, make, oracle_pairs, rel, sample_pairs, to_device, y_to_numpy

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_02_gb300 import build as cuda_build

    cuda_build.build()
    ssd.load_library()


def run(inp, flags=0, init=True, D=True):
    t = to_device(inp)
    y, fin = ssd.fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"] if D else None, chunk=inp.chunk,
                     init_state=t["init"] if init else None, flags=flags)
    torch.cuda.synchronize()
    return y_to_numpy(y), fin.cpu().numpy()


def check_against_oracle(inp, pairs=None, flags=0):
    y, fin = run(inp, flags)
    b, L, H, P = inp.x.shape
    if pairs is None:
        pairs = [(bb, hh) for bb in range(b) for hh in range(H)]
    out = oracle_pairs(inp, pairs)
    tol = TOL[inp.io_dtype]
    ey = rel(gather_y(y, pairs), out["y"])
    ef = rel(np.stack([fin[bb, hh] for bb, hh in pairs]), out["final"])
    assert ey <= tol and ef <= tol, "y err %.3e, final err %.3e (tol %.0e)" % (ey, ef, tol)
    return ey, ef


# ---------------------------------------------------------------- named workloads


def test_tiny_fp32_full():
    check_against_oracle(make("tiny_fp32"))


def test_mamba2_130m_layer_full():
    check_against_oracle(make("mamba2_130m_layer"))


def test_mamba2_2p7b_layer_sampled():
    inp = make("mamba2_2p7b_layer")
    check_against_oracle(inp, sample_pairs(2, 80, 6))


@pytest.mark.parametrize("n", [64, 128, 256, 512])
def test_state_size_sweep_sampled(n):
    inp = make("state_sweep_n%d" % n)
    check_against_oracle(inp, sample_pairs(1, 32, 4))


def test_long_256k_sampled_and_chained_segments():
    inp = make("long_256k")
    t = to_device(inp)
    y, fin = ssd.fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], chunk=256)
    # the same sequence as four 64K segments, each starting from the previous final state
    seg = 65536
    state = None
    ys = []
    for k in range(4):
        sl = slice(k * seg, (k + 1) * seg)
        yk, state = ssd.fwd(t["x"][:, sl].contiguous(), t["dt"][:, sl].contiguous(), t["A"],
                            t["B"][:, sl].contiguous(), t["C"][:, sl].contiguous(), t["D"], chunk=256,
                            init_state=state)
        ys.append(yk)
    torch.cuda.synchronize()
    y_np = y_to_numpy(y)
    fin_np = fin.cpu().numpy()
    ych = np.concatenate([y_to_numpy(v) for v in ys], axis=1)
    assert rel(ych, y_np) <= 2e-2 and rel(state.cpu().numpy(), fin_np) <= 2e-2
    pairs = [(0, 0), (0, 31)]
    out = oracle_pairs(inp, pairs)
    assert rel(gather_y(y_np, pairs), out["y"]) <= 2e-2
    assert rel(np.stack([fin_np[0, h] for _, h in pairs]), out["final"]) <= 2e-2
    assert rel(gather_y(ych, pairs), out["y"]) <= 2e-2


# ---------------------------------------------------------------- edge cases


EDGE = [
    dict(batch=2, seqlen=1000, nheads=6, headdim=64, dstate=128, chunk=256),   # ragged last chunk
    dict(batch=1, seqlen=100, nheads=4, headdim=64, dstate=128, chunk=256),    # L < Q/2: empty m-tile
    dict(batch=1, seqlen=1, nheads=3, headdim=64, dstate=64, chunk=256),       # one token
    dict(batch=2, seqlen=384, nheads=5, headdim=64, dstate=128, chunk=128),    # odd H, chunk 128
    dict(batch=1, seqlen=512, nheads=8, headdim=64, dstate=64, ngroups=2, chunk=256),  # groups
    dict(batch=1, seqlen=512, nheads=6, headdim=64, dstate=128, ngroups=2, chunk=256),  # 3 heads per group
    dict(batch=1, seqlen=300, nheads=3, headdim=32, dstate=48, chunk=64),      # CUDA-core path shapes
    dict(batch=1, seqlen=700, nheads=2, headdim=64, dstate=256, chunk=256),
    dict(batch=2, seqlen=600, nheads=3, headdim=64, dstate=384, chunk=128),   # wide state, Q = 128
    dict(batch=1, seqlen=520, nheads=4, headdim=64, dstate=256, ngroups=2, chunk=256),  # wide x groups
    dict(batch=1, seqlen=500, nheads=5, headdim=64, dstate=192, chunk=128),   # wide, 3 K steps
    dict(batch=1, seqlen=333, nheads=5, headdim=96, dstate=80, chunk=128),    # CUDA cores: ragged p tile
]


@pytest.mark.parametrize("shape", EDGE)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edge_shapes(shape, dtype):
    inp = synth.make_inputs(io_dtype=dtype, init=True, seed=3, **shape)
    check_against_oracle(inp)


@pytest.mark.parametrize("shape", [
    # odd heads per group (a pair with one head), two groups, ragged end
    dict(batch=1, seqlen=118000, nheads=6, headdim=64, dstate=128, ngroups=2, chunk=256),
    dict(batch=1, seqlen=117760, nheads=8, headdim=64, dstate=64, chunk=256),
], ids=["g2_odd_heads", "n64"])
def test_persistent_chunk_state_shapes(shape):
    # enough (head pair, n-tile, chunk) items for chunk_state's persistent kernel (a dozen or
    # more per SM); every head compared with the oracle over the whole sequence
    inp = synth.make_inputs(io_dtype="bf16", init=True, seed=41, **shape)
    check_against_oracle(inp)


@pytest.mark.parametrize("nheads,seqlen,chunk", [
    (32, 19520 + 37, 64), (48, 13056 + 101, 128),                        # one CTA per tile
    (32, 38912 + 37, 64), (16, 77824 + 5, 128), (8, 38912 + 61, 64),     # TMA-staged, persistent
], ids=["tile32_q64", "tile16_q128", "tma_tile32_q64", "tma_tile16_q128", "tma_tile8_q64"])
def test_cumsum_wide_head_tiles(nheads, seqlen, chunk):
    # chunk_cumsum with 32, 16 or 8 heads per tile (runs of 8 tokens per lane; 2 for 8 heads of a
    # 64-token chunk), in the one-CTA-per-tile kernel and, with four or more tiles per SM, the
    # persistent TMA kernel; ragged last chunk.  cs2 and dt checked directly, then y.
    inp = synth.make_inputs(batch=1, seqlen=seqlen, nheads=nheads, headdim=16, dstate=16, chunk=chunk,
                            io_dtype="f32", init=True, seed=17)
    t = to_device(inp)
    prob = ssd.problem_of(t["x"], t["B"], chunk)
    ws = ssd.alloc_workspace(prob)
    ssd.chunk_cumsum(prob, t["dt"], t["A"], ws)
    torch.cuda.synchronize()
    cs2, dtT = [v.float().cpu().numpy() for v in ssd.intermediates(prob, ws)[:2]]
    cs2_ref, dt_ref = ref.cumsum_log2(inp.dt, inp.A, chunk)
    assert rel(cs2, cs2_ref) <= 1e-6
    assert np.array_equal(dtT, dt_ref.astype(np.float32))
    # padded tokens of the last chunk repeat its last token's value exactly
    n_last = seqlen - (-(-seqlen // chunk) - 1) * chunk
    last = cs2[:, :, -1, :]
    assert np.array_equal(last[..., n_last:], np.repeat(last[..., n_last - 1:n_last], chunk - n_last, axis=-1))
    check_against_oracle(inp)


FUSED_SHAPES = [
    dict(batch=2, seqlen=1000, nheads=6, headdim=64, dstate=128, chunk=256),             # ragged
    dict(batch=1, seqlen=100, nheads=4, headdim=64, dstate=64, chunk=256),               # one chunk
    dict(batch=2, seqlen=384, nheads=5, headdim=64, dstate=128, chunk=128),              # odd H, Q 128
    dict(batch=1, seqlen=1536, nheads=6, headdim=64, dstate=128, ngroups=2, chunk=256),  # 3 heads / group
    dict(batch=3, seqlen=2300, nheads=8, headdim=64, dstate=64, ngroups=2, chunk=128),
]


@pytest.mark.parametrize("shape", FUSED_SHAPES)
@pytest.mark.parametrize("init", [True, False])
def test_fused_fwd_pass_state(shape, init):
    # chunk_state + state_passing as one kernel (forced): y and the final state against the oracle
    inp = synth.make_inputs(io_dtype="bf16", init=init, seed=29, **shape)
    y, fin = run(inp, flags=ssd.FLAG_FUSED_STATE, init=init)
    b, L, H, P = inp.x.shape
    pairs = [(bb, hh) for bb in range(b) for hh in range(H)]
    out = oracle_pairs(inp, pairs)
    assert rel(gather_y(y, pairs), out["y"]) <= 2e-2
    assert rel(np.stack([fin[bb, hh] for bb, hh in pairs]), out["final"]) <= 2e-2


@pytest.mark.parametrize("flags", [ssd.FLAG_FUSED_STATE, ssd.FLAG_SEPARATE_STATE_PASSING])
def test_fwd_pass_state_entry_point(flags):
    # ssd_fwd_pass_state fused or as two kernels: hprev (the state entering every chunk) and the
    # final state against the oracle's chunk inputs; the separate path's S against its chunk states
    inp = synth.make_inputs(batch=2, seqlen=1100, nheads=6, headdim=64, dstate=128, ngroups=2, chunk=256,
                            io_dtype="bf16", init=True, seed=31)
    t = to_device(inp)
    prob = ssd.problem_of(t["x"], t["B"], 256, flags)
    ws = ssd.alloc_workspace(prob)
    fin = torch.empty(2, 6, 64, 128, device="cuda")
    ssd.chunk_cumsum(prob, t["dt"], t["A"], ws)
    ssd.fwd_pass_state(prob, t["x"], t["B"], t["init"], fin, ws)
    assert ssd.read_status(ws) == 0
    assert bool(ssd.kernel_plan(prob) & 4) == (flags == ssd.FLAG_FUSED_STATE)
    _, _, S, hprev = [v.float().cpu().numpy() for v in ssd.intermediates(prob, ws)]
    pairs = [(b, h) for b in range(2) for h in range(6)]
    out = oracle_pairs(inp, pairs, want_chunk_in=True)
    assert rel(np.stack([hprev[b, :, h] for b, h in pairs]), out["chunk_in"]) <= 1e-2
    assert rel(np.stack([fin.cpu().numpy()[b, h] for b, h in pairs]), out["final"]) <= 1e-2
    if flags == ssd.FLAG_SEPARATE_STATE_PASSING:
        S_ref = ref.chunk_states(inp.x, inp.dt, inp.A, inp.B, 256)      # every (b, h) in order
        assert rel(np.stack([S[b, :, h] for b, h in pairs]), S_ref) <= 1e-2


def test_slow_decay_exercises_state_passing():
    # |A| in [0.001, 0.05]: the state carries across many chunks
    inp = synth.make_inputs(batch=1, seqlen=4096, nheads=4, headdim=64, dstate=128, chunk=256,
                            io_dtype="bf16", init=True, seed=5, a_range=(0.001, 0.05))
    check_against_oracle(inp)


# ---------------------------------------------------------------- large steps
#
# The recurrence holds for any positive step and negative A; the kernels factor each decay
# weight 2^{cs2_i - cs2_j} dt_j into per-row and per-column parts, which must stay inside
# float32's range however fast the state decays.  dt in [0.5, 2] with A = -16 decays by
# 2^-11.5 .. 2^-46 per token (hundreds of log2 units per 32-token block); dt in [0.05, 0.3]
# with A = -4 puts a block's decay span around the point where the diagonal block switches
# from factored to per-element weights.

BIG_STEPS = dict(dt_mean=0.5, dt_clip=(0.5, 2.0), a_range=(16.0, 16.0))
MID_STEPS = dict(dt_mean=-2.0, dt_clip=(0.05, 0.3), a_range=(4.0, 4.0))


@pytest.mark.parametrize("steps", [BIG_STEPS, MID_STEPS], ids=["big", "mid"])
@pytest.mark.parametrize("shape", [
    dict(batch=1, seqlen=1000, nheads=4, headdim=64, dstate=128, chunk=256),   # tensor-core scan
    dict(batch=1, seqlen=700, nheads=3, headdim=64, dstate=256, chunk=256),    # two state slices
    dict(batch=1, seqlen=600, nheads=2, headdim=64, dstate=128, chunk=128),
    dict(batch=1, seqlen=520, nheads=3, headdim=64, dstate=128, chunk=64),     # CUDA-core scan
], ids=["q256n128", "q256n256", "q128n128", "q64n128"])
def test_large_steps_bf16(shape, steps):
    inp = synth.make_inputs(io_dtype="bf16", init=True, seed=21, **shape, **steps)
    check_against_oracle(inp)


@pytest.mark.parametrize("steps", [BIG_STEPS, MID_STEPS], ids=["big", "mid"])
@pytest.mark.parametrize("chunk", [64, 256])
def test_large_steps_f32_cuda_cores(chunk, steps):
    inp = synth.make_inputs(batch=1, seqlen=600, nheads=3, headdim=32, dstate=64, chunk=chunk,
                            io_dtype="f32", init=True, seed=22, **steps)
    check_against_oracle(inp)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_large_steps_forced_onto_cuda_cores(dtype):
    inp = synth.make_inputs(batch=1, seqlen=1000, nheads=4, headdim=64, dstate=128, chunk=256,
                            io_dtype=dtype, init=True, seed=23, **BIG_STEPS)
    check_against_oracle(inp, flags=ssd.FLAG_FORCE_SIMT)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_one_head_with_large_steps_among_small(dtype):
    # heads 0, 1, 3 keep the workloads' steps; head 2 takes steps in [0.5, 2] with A = -16
    inp = synth.make_inputs(batch=2, seqlen=900, nheads=4, headdim=64, dstate=128, chunk=256,
                            io_dtype=dtype, init=True, seed=24)
    big = synth.make_inputs(batch=2, seqlen=900, nheads=4, headdim=64, dstate=128, chunk=256,
                            io_dtype=dtype, init=True, seed=25, **BIG_STEPS)
    inp.dt[:, :, 2] = big.dt[:, :, 2]
    inp.A[2] = big.A[2]
    check_against_oracle(inp)
    # the heads with ordinary steps are held to the tolerance on their own
    y, _ = run(inp)
    pairs = [(b, h) for b in range(2) for h in (0, 1, 3)]
    out = oracle_pairs(inp, pairs)
    assert rel(gather_y(y, pairs), out["y"]) <= TOL[dtype]


def test_no_D_and_no_init():
    inp = synth.make_inputs(batch=1, seqlen=512, nheads=4, headdim=64, dstate=128, chunk=256,
                            io_dtype="bf16", init=False, seed=7, with_D=False)
    check_against_oracle(inp)


def test_tensor_core_and_cuda_core_paths_agree():
    inp = synth.make_inputs(batch=2, seqlen=1024, nheads=4, headdim=64, dstate=128, chunk=256,
                            io_dtype="bf16", init=True, seed=11)
    y_tc, f_tc = run(inp)
    y_sc, f_sc = run(inp, flags=ssd.FLAG_FORCE_SIMT)
    assert rel(y_tc, y_sc) <= 2e-2 and rel(f_tc, f_sc) <= 2e-2


@pytest.mark.parametrize("n", [256, 512])
def test_wide_tensor_core_scan_matches_cuda_core(n):
    # state sizes above 128: the readout kernel, then chunk_scan with a K loop over the state
    inp = synth.make_inputs(batch=1, seqlen=1000, nheads=4, headdim=64, dstate=n, chunk=256,
                            io_dtype="bf16", init=True, seed=13)
    y_tc, f_tc = run(inp)
    y_sc, f_sc = run(inp, flags=ssd.FLAG_FORCE_SIMT)
    assert rel(y_tc, y_sc) <= 2e-2 and rel(f_tc, f_sc) <= 2e-2


def test_repeat_runs_are_bitwise_identical():
    inp = make("mamba2_130m_layer")
    y1, f1 = run(inp)
    y2, f2 = run(inp)
    assert np.array_equal(y1, y2) and np.array_equal(f1, f2)


# ---------------------------------------------------------------- per-step intermediates


@pytest.mark.parametrize("flags", [0, ssd.FLAG_FORCE_SIMT])
def test_step_intermediates(flags):
    inp = synth.make_inputs(batch=2, seqlen=900, nheads=4, headdim=64, dstate=128, chunk=256,
                            io_dtype="bf16", init=True, seed=13)
    t = to_device(inp)
    prob = ssd.problem_of(t["x"], t["B"], 256, flags)
    ws = ssd.alloc_workspace(prob)
    fin = torch.empty(2, 4, 64, 128, device="cuda")
    y = torch.empty_like(t["x"])
    ssd.chunk_cumsum(prob, t["dt"], t["A"], ws)
    ssd.chunk_state(prob, t["x"], t["B"], ws)
    ssd.state_passing(prob, t["init"], fin, ws)
    ssd.chunk_scan(prob, t["x"], t["B"], t["C"], t["D"], y, ws)
    assert ssd.read_status(ws) == 0
    cs2, dtT, S, hprev = [v.float().cpu().numpy() for v in ssd.intermediates(prob, ws)]
    cs2_ref, dt_ref = ref.cumsum_log2(inp.dt, inp.A, 256)
    assert rel(cs2, cs2_ref) <= 1e-6
    assert np.array_equal(dtT, dt_ref.astype(np.float32))
    pairs = [(b, h) for b in range(2) for h in range(4)]
    S_ref = ref.chunk_states(inp.x, inp.dt, inp.A, inp.B, 256)          # (8, nc, P, N)
    got_S = np.stack([S[b, :, h] for b, h in pairs])
    assert rel(got_S, S_ref) <= 1e-2
    out = oracle_pairs(inp, pairs, want_chunk_in=True)
    got_h = np.stack([hprev[b, :, h] for b, h in pairs])
    assert rel(got_h, out["chunk_in"]) <= 1e-2
    assert rel(np.stack([fin.cpu().numpy()[b, h] for b, h in pairs]), out["final"]) <= 1e-2
    assert rel(gather_y(y_to_numpy(y), pairs), out["y"]) <= 2e-2


def test_f32_intermediates_are_tight():
    inp = make("tiny_fp32")
    t = to_device(inp)
    prob = ssd.problem_of(t["x"], t["B"], inp.chunk)
    ws = ssd.alloc_workspace(prob)
    y, fin = ssd.fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], chunk=inp.chunk, workspace=ws)
    cs2, dtT, S, hprev = [v.cpu().numpy() for v in ssd.intermediates(prob, ws)]
    S_ref = ref.chunk_states(inp.x, inp.dt, inp.A, inp.B, inp.chunk)
    out = oracle_pairs(inp, [(0, h) for h in range(4)], want_chunk_in=True)
    assert rel(np.stack([S[0, :, h] for h in range(4)]), S_ref) <= 1e-4
    assert rel(np.stack([hprev[0, :, h] for h in range(4)]), out["chunk_in"]) <= 1e-4


# ---------------------------------------------------------------- failure detection


def test_bounded_wait_reports_timeout_and_context_survives():
    word = torch.zeros(4, dtype=torch.int32, device="cuda")
    ssd.selftest_wait_timeout(word, 2_000_000)   # 2 ms on a barrier nothing completes
    assert ssd.read_status(word) == 5            # SSD_ERR_TIMEOUT
    check_against_oracle(make("tiny_fp32"))      # the context is still usable
