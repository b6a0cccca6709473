"""SSD forward-scan benchmark: tokens/s on GB300 through the library's C ABI.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one ssd_fwd call: the whole forward scan (chunk_cumsum, chunk_state, state_passing,
chunk_scan) over one batch of seeded synthetic input already resident in HBM.  L2 is flushed (a
256 MiB write and a 256 MiB read, outside the timed events) before every timed step.  The step
time comes from CUDA events around the call; per-kernel times (for the roofline) from a second
pass through the four per-step entry points (the same launches) with an event between them.
``--impl reference`` times the float64 CPU oracle instead, on a bounded sample of the same
workload.  Rank 0 prints one JSON line.

Workloads named ``decode_*`` time the recurrent form instead (ssd_decode): one step is one
launch that advances the resident float32 state of every (batch, head) by ``seqlen`` tokens;
the metric is decoded tokens/s and the roofline is HBM (the state is read and written once).
"""
import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "long_256k"
METRIC = "SSD forward tokens/s on 1 GB300 + per-kernel % of HBM/tensor roofline"
METRIC_DECODE = "SSD decode tokens/s on 1 GB300 + % of HBM roofline"


METRIC_SEL = "Mamba-1 selective scan tokens/s on 1 GB300 + % of exp (MUFU) roofline"
# one ex2 per (batch, token, channel, state) is the method's irreducible special-function work;
# GB300: 152 SMs x 32 MUFU results per clock (one warp instruction per SM per clock: the XU
# pipe's peak as ncu accounts it) x 2.07 GHz, in G/s
MUFU_PEAK_GPS = 152 * 32 * 2.07


def is_decode(workload):
    return workload.startswith("decode")


def is_selective(workload):
    return workload.startswith("mamba1_")


METRIC_BWD = "SSD backward tokens/s on 1 GB300 + % of HBM roofline"


def is_bwd(workload):
    return workload.startswith("bwd_")


def metric_of(workload):
    if is_selective(workload):
        return METRIC_SEL
    if is_bwd(workload):
        return METRIC_BWD
    return METRIC_DECODE if is_decode(workload) else METRIC


def algorithmic_bwd(shape):
    """Minimum HBM bytes of one backward pass: x, dt, B, C, dy (and init, dfinal) read once,
    dx, ddt, dB, dC (and dinit) written once; A, D, dA, dD are negligible."""
    b, L, H, P, N, G = (shape[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups"))
    e = 2 if shape["io_dtype"] == "bf16" else 4
    st = b * H * P * N * 4
    return 3 * b * L * H * P * e + 4 * b * L * G * N * e + 2 * b * L * H * 4 + 2 * st + (st if shape["init"] else 0)
KERNELS = ("chunk_cumsum", "chunk_state", "state_passing", "chunk_scan")
KERNELS_FUSED = ("chunk_cumsum", "fwd_pass_state", "chunk_scan")   # chunk_state + state_passing in one


def step_kernels(plan):
    """The kernels of one forward step for an ssd_kernel_plan value (bit 2: fused fwd_pass_state)."""
    return KERNELS_FUSED if plan >= 0 and plan & 4 else KERNELS


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="approximate CPU time budget of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


# ----------------------------------------------------------------------------- accounting


def algorithmic(shape):
    """Minimum HBM bytes and useful FLOPs per launch of each kernel (the roofline inputs)."""
    b, L, H, P, N, G, Q = (shape[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate",
                                               "ngroups", "chunk"))
    e = 2 if shape["io_dtype"] == "bf16" else 4
    nc = -(-L // Q)
    st = b * nc * H * P * N                      # elements of S / hprev
    cs = b * H * nc * Q * 4                      # bytes of one cs2 / dtT array
    by = {
        "chunk_cumsum": b * L * H * 4 + H * 4 + 2 * cs,
        "chunk_state": b * L * H * P * e + b * L * G * N * e + 2 * cs + st * e,
        "state_passing": st * e + b * H * nc * 4 + st * e + 2 * b * H * P * N * 4,
        "chunk_scan": 2 * b * L * H * P * e + 2 * b * L * G * N * e + 2 * cs + st * e + H * 4,
        # the fused kernel: x, B, cs2 / dtT in, hprev and the final state out (S stays on chip)
        "fwd_pass_state": b * L * H * P * e + b * L * G * N * e + 2 * cs + st * e + b * H * P * N * 4,
    }
    fl = {
        "chunk_cumsum": 2 * b * L * H,
        "chunk_state": 2 * b * nc * H * Q * P * N,
        "state_passing": 2 * st,
        "fwd_pass_state": 2 * b * nc * H * Q * P * N + 2 * st,
        "chunk_scan": (2 * b * nc * G * (Q * (Q + 1) // 2) * N + 2 * b * nc * H * (Q * (Q + 1) // 2) * P
                       + 2 * b * nc * H * Q * P * N),
    }
    if shape["init"]:
        by["state_passing"] += b * H * P * N * 4
        by["fwd_pass_state"] += b * H * P * N * 4
    return by, fl


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm=float(pk["hbm_gbs"]), bf16=float(pk["bf16_tflops"]),
                    bf16_sus=float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def source_digest(kernel):
    """Digest of a kernel's source file with comments and whitespace removed: a profile stays
    valid across comment edits and is dropped by any change to the code."""
    files = {"chunk_cumsum": "chunk_cumsum.cu", "chunk_state": "chunk_state_tc.cu",
             "fwd_pass_state": "chunk_state_tc.cu",
             "state_passing": "state_passing.cu", "chunk_scan": "chunk_scan_tc.cu",
             "decode": "decode.cu", "selective_scan": "selective_scan.cu"}
    p = os.path.join(ROOT, "state_space_model_02_gb300", "csrc", files[kernel])
    with open(p) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = "".join(text.split())
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if its kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "%s__%s.txt" % (kernel, workload))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"^dram_bytes_per_launch\s*=\s*([0-9.eE+]+)", text, re.M)
    h = re.search(r"^source_sha256_16\s*=\s*([0-9a-f]+)", text, re.M)
    if not m or not h or h.group(1) != source_digest(kernel):
        return None
    return float(m.group(1))


# ------------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------- CPU baseline


def algorithmic_decode(shape):
    """Minimum HBM bytes and FLOPs of one decode launch: the state read and written once
    (float32), each token's x, dt, B, C read and y written once, A and D read once."""
    b, T, H, P, N, G = (shape[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups"))
    e = 2 if shape["io_dtype"] == "bf16" else 4
    by = 2 * b * H * P * N * 4 + b * T * (2 * H * P * e + 2 * G * N * e + H * 4) + 2 * H * 4
    fl = b * T * H * P * (4 * N + 2)   # update (2 per element) + C contraction (2) + D x
    return by, fl


def cpu_baseline_selective(inp, budget_s):
    """The float64 selective-scan oracle on the host cores over a bounded sample: whole
    sequences of as many channels as fit the time budget (tokens scaled to the layer)."""
    from oracle import ref, selective

    b, L, D = inp.x.shape
    threads = ref.num_threads()

    def run(nch):
        sub = lambda a: np.ascontiguousarray(a[:, :, :nch])
        t0 = time.perf_counter()
        selective.selective_scan(sub(inp.x), sub(inp.delta), inp.A[:nch], inp.B, inp.C, inp.D[:nch],
                                 None if inp.init is None else np.ascontiguousarray(inp.init[:, :nch]))
        return time.perf_counter() - t0

    probe = min(D, max(threads, 8))
    per_ch = run(probe) / probe
    nch = int(min(D, max(probe, budget_s / max(per_ch, 1e-9))))
    reps, el = 0, 0.0
    while reps == 0 or (el < budget_s and reps < 100):
        el += run(nch)
        reps += 1
    tokens = reps * b * L * nch / D
    return {"value": tokens / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d channels x %d sequences of %d tokens x %d passes, float64, %.1f s"
                      % (nch, D, b, L, reps, el)}


def cpu_baseline_bwd(inp, dy, dfin, budget_s):
    """The float64 adjoint oracle on the host over a bounded sample: whole sequences of as many
    (batch 0) heads as fit the budget, tokens scaled to the layer."""
    from oracle.ref_bwd import recurrence_bwd_np

    b, L, H, P = inp.x.shape
    G = inp.B.shape[2]
    hpg = H // G

    def run(nh):
        sl = lambda a: np.ascontiguousarray(a[:1, :, :nh])
        gsel = 1
        t0 = time.perf_counter()
        recurrence_bwd_np(sl(inp.x), np.ascontiguousarray(inp.dt[:1, :, :nh]), inp.A[:nh],
                          np.ascontiguousarray(inp.B[:1, :, :gsel]), np.ascontiguousarray(inp.C[:1, :, :gsel]),
                          inp.D[:nh], None if inp.init is None else np.ascontiguousarray(inp.init[:1, :nh]),
                          np.ascontiguousarray(dy[:1, :, :nh]), np.ascontiguousarray(dfin[:1, :nh]))
        return time.perf_counter() - t0

    nh = min(2, H)   # two heads of group 0: the NumPy oracle's cost grows with heads x tokens
    reps, el = 0, 0.0
    while reps == 0 or (el < budget_s and reps < 100):
        el += run(nh)
        reps += 1
    tokens = reps * L * nh / H   # whole-layer tokens of one sequence the sample amounts to
    return {"value": tokens / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "%d of %d heads of one sequence of %d tokens x %d passes, float64 adjoint "
                      "recurrence (NumPy), %.1f s" % (nh, H, L, reps, el)}


def cpu_baseline(inp, budget_s):
    """The float64 oracle as it stands, on the host cores, over a bounded sample of the
    workload: whole (batch, head) sequences, as many as fit the time budget."""
    from oracle import ref

    b, L, H, P = inp.x.shape
    pairs = [(bb, hh) for bb in range(b) for hh in range(H)]
    threads = ref.num_threads()
    # probe one pair per thread, then size the sample to the budget
    probe = pairs[:max(1, min(len(pairs), threads))]
    t0 = time.perf_counter()
    ref.recurrence(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, chunk=inp.chunk,
                   pairs=np.array(probe), want_final=True)
    dt_probe = time.perf_counter() - t0
    per_pair = dt_probe / len(probe)
    n = int(min(len(pairs), max(len(probe), budget_s / max(per_pair, 1e-9))))
    n = max(threads, (n // threads) * threads) if n >= threads else n
    n = min(n, len(pairs))
    sample = pairs[:n]
    reps, el = 0, 0.0
    while reps == 0 or (el < budget_s and reps < 100):   # repeat small workloads up to the budget
        t0 = time.perf_counter()
        ref.recurrence(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, chunk=inp.chunk,
                       pairs=np.array(sample), want_final=True)
        el += time.perf_counter() - t0
        reps += 1
    tokens = reps * b * L * (len(sample) / (b * H))  # whole-layer tokens the sample amounts to
    return {"value": tokens / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d (batch, head) sequences of %d tokens x %d passes, float64 "
                      "recurrence, %.1f s" % (len(sample), b * H, L, reps, el)}


# ------------------------------------------------------------------------------ arms


def max_over_ranks(ms, ws, dist, dev):
    """The job's time for a quantity every rank measured: the slowest rank's (MAX all-reduce)."""
    if ws <= 1:
        return float(ms)
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(tokens_per_rank, ws, ms):
    """Whole-job throughput: every rank's tokens over the job's (slowest rank's) time."""
    return ws * tokens_per_rank / (ms * 1e-3)


def pipelined_e2e(torch, dev, steps, pin, compute, warmup=3):
    """End-to-end time per step through the public API, host buffers in and out.

    Every step uploads its inputs from pinned host memory, computes, and reads its outputs back
    into pinned host memory.  Steps are pipelined the way a serving loop runs them: three
    streams (upload, compute, download) and two buffer sets, so step k+1's upload and step
    k-1's download overlap step k's compute.  compute(dev_inputs, slot) runs on the current
    (compute) stream and returns the device tensors to download.  Returns (ms per step,
    bytes uploaded per step, bytes downloaded per step); the timed region starts empty (after a
    synchronize) and ends when the last download has landed.
    """
    s_up, s_cmp, s_down = (torch.cuda.Stream(dev) for _ in range(3))
    dev_in = [{k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in pin.items()}
              for _ in range(2)]
    host_out = [None, None]
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("up", "cmp", "down")}
    d2h = [0]

    def one(k):
        i = k % 2
        with torch.cuda.stream(s_up):
            if k >= 2:
                s_up.wait_event(ev["cmp"][i])   # slot i's inputs are no longer read
            for name, v in pin.items():
                if v is not None:
                    dev_in[i][name].copy_(v, non_blocking=True)
            ev["up"][i].record(s_up)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev["up"][i])
            if k >= 2:
                s_cmp.wait_event(ev["down"][i])  # slot i's outputs have been read back
            outs = [o for o in compute(dev_in[i], i) if o is not None]
            ev["cmp"][i].record(s_cmp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev["cmp"][i])
            if host_out[i] is None:
                host_out[i] = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
            for o, h in zip(outs, host_out[i]):
                o.record_stream(s_down)
                h.copy_(o, non_blocking=True)
            d2h[0] = sum(o.numel() * o.element_size() for o in outs)
            ev["down"][i].record(s_down)

    for k in range(warmup):
        one(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    for k in range(warmup, warmup + steps):
        one(k)
    e1.record(s_down)
    torch.cuda.synchronize()
    h2d = sum(v.numel() * v.element_size() for v in pin.values() if v is not None)
    return e0.elapsed_time(e1) / steps, h2d, d2h[0]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from state_space_model_02_gb300 import synth

    if is_bwd(args.workload):
        base_wl = args.workload[len("bwd_"):]
        inp = synth.make_config(base_wl, seed=args.seed)
        shape = dict(synth.CONFIGS[base_wl])
        rng = np.random.default_rng(args.seed + 1)
        b_, L_, H_, P_ = inp.x.shape
        dy_ = rng.standard_normal((b_, L_, H_, P_)).astype(np.float32)
        df_ = rng.standard_normal((b_, H_, P_, inp.B.shape[3])).astype(np.float32)
        baseline = lambda i, budget: cpu_baseline_bwd(i, dy_, df_, budget)
    elif is_selective(args.workload):
        inp = synth.make_selective_config(args.workload, seed=args.seed)
        shape = dict(synth.SELECTIVE_CONFIGS[args.workload])
        baseline = cpu_baseline_selective
    else:
        inp = synth.make_config(args.workload, seed=args.seed)
        shape = dict(synth.CONFIGS[args.workload])
        baseline = cpu_baseline
    vals = []
    per = max(1.0, args.cpu_seconds / max(1, args.steps))
    base = None
    for _ in range(args.steps):
        base = baseline(inp, per)
        vals.append(base["value"])
    v = float(np.median(vals))
    tokens = shape["batch"] * shape["seqlen"]
    line = {"impl": "reference", "metric": metric_of(args.workload), "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tokens / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, **shape},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": base["cores"], "kind": "oracle",
                             "sample": base["sample"]},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    from state_space_model_02_gb300 import build as cuda_build
    from state_space_model_02_gb300 import ssd, synth

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cuda_build.build()
    ssd.load_library()

    if is_selective(args.workload):
        return run_selective(args, torch, dist, ssd, synth, ws, rank, local, dev)
    if is_bwd(args.workload):
        return run_bwd(args, torch, dist, ssd, synth, ws, rank, local, dev)
    shape = dict(synth.CONFIGS[args.workload])
    inp = synth.make_config(args.workload, seed=args.seed)
    bf16 = inp.io_dtype == "bf16"

    def io(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else np.ascontiguousarray(a))
        return t.view(torch.bfloat16) if bf16 else t

    host = dict(x=io(inp.x), dt=torch.from_numpy(inp.dt), A=torch.from_numpy(inp.A), B=io(inp.B),
                C=io(inp.C), D=torch.from_numpy(inp.D),
                init=None if inp.init is None else torch.from_numpy(inp.init))
    d = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    if is_decode(args.workload):
        return run_decode(args, torch, dist, ssd, ws, rank, local, dev, shape, inp, host, d)
    prob = ssd.problem_of(d["x"], d["B"], inp.chunk)
    wsbuf = ssd.alloc_workspace(prob, dev)
    y = torch.empty_like(d["x"])
    fin = torch.empty((prob.batch, prob.nheads, prob.headdim, prob.dstate), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2(k):
        # write a buffer larger than L2, then read another one, so the timed step starts with
        # neither its own data nor dirty lines left to write back in L2
        flush.fill_(k & 0xFF)
        flush_rd.max()  # a plain read of the buffer (no dtype conversion pass)
    stream = torch.cuda.current_stream(dev)

    def step():
        # one ssd_fwd call: chunk_cumsum, chunk_state and state_passing (one fused fwd_pass_state
        # kernel where the plan says so), chunk_scan, launched back to back
        ssd.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], chunk=inp.chunk, init_state=d["init"],
                y=y, final_state=fin, workspace=wsbuf, stream=stream)

    plan = ssd.kernel_plan(prob)
    kernels = step_kernels(plan)

    def step_by_kernel(evs):
        # the same launches through the per-step entry points, an event between launches
        calls = {
            "chunk_cumsum": lambda: ssd.chunk_cumsum(prob, d["dt"], d["A"], wsbuf, stream),
            "chunk_state": lambda: ssd.chunk_state(prob, d["x"], d["B"], wsbuf, stream),
            "state_passing": lambda: ssd.state_passing(prob, d["init"], fin, wsbuf, stream),
            "fwd_pass_state": lambda: ssd.fwd_pass_state(prob, d["x"], d["B"], d["init"], fin, wsbuf, stream),
            "chunk_scan": lambda: ssd.chunk_scan(prob, d["x"], d["B"], d["C"], d["D"], y, wsbuf, stream),
        }
        for i, n in enumerate(kernels):
            if evs:
                evs[i].record(stream)
            calls[n]()
        if evs:
            evs[len(kernels)].record(stream)

    for k in range(max(3, args.warmup)):
        flush_l2(k)
        step()
    torch.cuda.synchronize()
    status = ssd.read_status(wsbuf, stream)
    if status != 0:
        raise RuntimeError("kernel status %d during warm-up" % status)

    clocks = ClockSampler(local)
    # the step: one ssd_fwd call, its launches back to back (programmatic dependent launch lets
    # each kernel's prologue overlap its predecessor), bracketed by one pair of events
    step_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for k in range(args.steps):
        flush_l2(k)                   # evict L2: untimed, outside the step's events
        step_evs[k][0].record(stream)
        step()
        step_evs[k][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    totals = [e[0].elapsed_time(e[1]) for e in step_evs]
    ms_step = float(np.sum(totals) / args.steps)
    # per-kernel durations (for the roofline): the same steps again with an event between kernels
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush_l2(k)
        step_by_kernel(evs[k])
    torch.cuda.synchronize()
    per_kernel = {n: [] for n in kernels}
    for e in evs:
        for i, n in enumerate(kernels):
            per_kernel[n].append(e[i].elapsed_time(e[i + 1]))
    ms_step = max_over_ranks(ms_step, ws, dist, dev)
    tokens = prob.batch * prob.seqlen
    value = job_rate(tokens, ws, ms_step)

    # roofline of every kernel; the dominant (largest share) is reported
    by, fl = algorithmic(shape)
    peaks = load_peaks()
    kern = {}
    for n in kernels:
        ms = float(np.mean(per_kernel[n]))
        t_hbm = by[n] / (peaks["hbm"] * 1e9)
        t_ten = fl[n] / (peaks["bf16"] * 1e12) if n in ("chunk_state", "fwd_pass_state", "chunk_scan") else 0.0
        bound = "hbm" if t_hbm >= t_ten else "tensor"
        ach = by[n] / (ms * 1e-3) / 1e9 if bound == "hbm" else fl[n] / (ms * 1e-3) / 1e12
        peak = peaks["hbm"] if bound == "hbm" else peaks["bf16"]
        kern[n] = {"us": 1e3 * ms, "share": ms / ms_step, "bound": bound, "achieved": ach, "peak": peak,
                   "frac": ach / peak, "alg_bytes": by[n], "alg_flops": fl[n],
                   "tensor_frac_of_peak": fl[n] / (ms * 1e-3) / 1e12 / peaks["bf16"]}
    dom = max(kernels, key=lambda n: kern[n]["us"])
    kd = kern[dom]
    tr = profiled_traffic(dom, args.workload)
    roofline = {"kernel": dom, "bound": kd["bound"], "achieved": kd["achieved"], "peak": kd["peak"],
                "unit": "GB/s" if kd["bound"] == "hbm" else "TFLOP/s", "frac": kd["frac"],
                "traffic": tr, "peak_source": peaks["src"] + " (MEASURED_PEAKS.json burst)"
                if peaks["src"] == "measured" else "fallback"}

    # end to end through the public API: pinned host in, result back to pinned host
    e2e = None
    if not args.no_e2e:
        pin = {k: (None if v is None else v.pin_memory()) for k, v in host.items()}
        ys = [y, torch.empty_like(y)]
        fins = [fin, torch.empty_like(fin)]

        def fwd_slot(src, i):
            return ssd.fwd(src["x"], src["dt"], src["A"], src["B"], src["C"], src["D"], chunk=inp.chunk,
                           init_state=src["init"], y=ys[i], final_state=fins[i], workspace=wsbuf)

        ms_e2e, h2d, d2h = pipelined_e2e(torch, dev, args.steps, pin, fwd_slot)
        ms_e2e = max_over_ranks(ms_e2e, ws, dist, dev)
        e2e = {"value": job_rate(tokens, ws, ms_e2e), "unit": "tokens/s", "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipelined": "upload / compute / download streams, two buffer sets"}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline(inp, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16 else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": args.workload, **shape,
                   "l2": "flushed before every step (256 MiB write + 256 MiB read, outside the timed events)",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "tensor_core_steps": {"chunk_state": bool(plan & 1), "chunk_scan": bool(plan & 2),
                                         "fused_fwd_pass_state": bool(plan & 4)}},
        "roofline": roofline,
        "kernels": {n: {k: (round(v, 4) if isinstance(v, float) else v) for k, v in kern[n].items()}
                    for n in kernels},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
        "gpu_launches": (len(kernels) - 1 + scan_launches(shape, plan)) * args.steps,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def scan_launches(shape, plan):
    """Launches of the chunk_scan step: with states above 128 columns the tensor-core path runs
    the readout kernel (the term through the chunk-start state) before chunk_scan."""
    n, q = shape["dstate"], shape["chunk"]
    return 2 if (plan & 2) and n > 128 and n % 64 == 0 and n >= q else 1


def run_bwd(args, torch, dist, ssd, synth, ws, rank, local, dev):
    """The backward arm: one ssd_bwd call per step (it runs the forward again inside)."""
    base_wl = args.workload[len("bwd_"):]
    shape = dict(synth.CONFIGS[base_wl])
    inp = synth.make_config(base_wl, seed=args.seed)
    bf16 = inp.io_dtype == "bf16"
    rng = np.random.default_rng(args.seed + 1)
    b, L, H, P = inp.x.shape
    N = inp.B.shape[3]
    dy_np = rng.standard_normal((b, L, H, P)).astype(np.float32)
    df_np = rng.standard_normal((b, H, P, N)).astype(np.float32)
    if bf16:
        dy_np = synth.to_bf16_bits(dy_np)

    def io(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else np.ascontiguousarray(a))
        return t.view(torch.bfloat16) if bf16 else t

    host = dict(x=io(inp.x), dt=torch.from_numpy(inp.dt), A=torch.from_numpy(inp.A), B=io(inp.B), C=io(inp.C),
                D=torch.from_numpy(inp.D), init=None if inp.init is None else torch.from_numpy(inp.init),
                dy=io(dy_np), dfin=torch.from_numpy(df_np))
    d = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    prob = ssd.problem_of(d["x"], d["B"], inp.chunk)
    wsbuf = torch.empty(ssd.load_library().ssd_bwd_workspace_bytes(ctypes_byref(prob)), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(k):
        flush.fill_(k & 0xFF)
        flush_rd.max()

    def step(src=d):
        return ssd.bwd(src["x"], src["dt"], src["A"], src["B"], src["C"], src["D"], src["dy"], chunk=inp.chunk,
                       init_state=src["init"], dfinal=src["dfin"], workspace=wsbuf, stream=stream)

    for k in range(max(3, args.warmup)):
        flush_l2(k)
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for k in range(args.steps):
        flush_l2(k)
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    ms_step = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    ms_step = max_over_ranks(ms_step, ws, dist, dev)
    tokens = b * L
    value = job_rate(tokens, ws, ms_step)
    by = algorithmic_bwd(shape)
    peaks = load_peaks()
    ach = by / (ms_step * 1e-3) / 1e9
    roofline = {"kernel": "ssd_bwd (whole pass)", "bound": "hbm", "achieved": ach, "peak": peaks["hbm"],
                "unit": "GB/s", "frac": ach / peaks["hbm"], "traffic": None,
                "peak_source": peaks["src"] + " (MEASURED_PEAKS.json burst)" if peaks["src"] == "measured" else "fallback"}

    e2e = None
    if not args.no_e2e:
        pin = {k: (None if v is None else v.pin_memory()) for k, v in host.items()}

        def bwd_slot(src, i):
            g = ssd.bwd(src["x"], src["dt"], src["A"], src["B"], src["C"], src["D"], src["dy"], chunk=inp.chunk,
                        init_state=src["init"], dfinal=src["dfin"], workspace=wsbuf)
            return [g[k] for k in sorted(g)]

        ms_e2e, h2d, d2h = pipelined_e2e(torch, dev, args.steps, pin, bwd_slot)
        ms_e2e = max_over_ranks(ms_e2e, ws, dist, dev)
        e2e = {"value": job_rate(tokens, ws, ms_e2e), "unit": "tokens/s", "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipelined": "upload / compute / download streams, two buffer sets"}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        dyf = synth.bf16_bits_to_f32(dy_np) if bf16 else dy_np
        cpu = cpu_baseline_bwd(inp, dyf, df_np, args.cpu_seconds)
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16 else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload; dy, dfinal ~ N(0, 1))",
        "config": {"workload": args.workload, **shape,
                   "l2": "flushed before every step (256 MiB write + 256 MiB read, outside the timed events)",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": roofline,
        "kernels": {"ssd_bwd": {"us": 1e3 * ms_step, "share": 1.0, "alg_bytes": by}},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "gpu_launches": bwd_launches(shape) * args.steps,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def bwd_launches(shape):
    """Kernel launches of one ssd_bwd call (dfinal given, dD and dinit wanted): two scans of 4
    launches with their input copies and the scalar steps, then the role-swapped scan pairs,
    one pair per 64-column slice when bf16 with headdim 64 (else one pair)."""
    P, N = shape["headdim"], shape["dstate"]
    init = 1 if shape["init"] else 0
    kw = 64 if shape["io_dtype"] == "bf16" and P == 64 and N % 64 == 0 else N
    head = 3 + 4 + 3 + 1 + 4 + 1 + 1 + 1 + 2 + init          # widen, scan, flips, decays, scan, combine, ...
    per_slice = (1 + init + 4 + 1) + (1 + 1 + 4 + 1)
    return head + 2 + (N // kw) * per_slice


def ctypes_byref(prob):
    import ctypes

    return ctypes.byref(prob.c_shape())


def run_selective(args, torch, dist, ssd, synth, ws, rank, local, dev):
    """The Mamba-1 arm: one ssd_selective_scan launch per step over resident inputs."""
    shape = dict(synth.SELECTIVE_CONFIGS[args.workload])
    inp = synth.make_selective_config(args.workload, seed=args.seed)
    bf16 = inp.io_dtype == "bf16"

    def io(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else np.ascontiguousarray(a))
        return t.view(torch.bfloat16) if bf16 else t

    host = dict(x=io(inp.x), delta=io(inp.delta), B=io(inp.B), C=io(inp.C))
    d = {k: v.to(dev) for k, v in host.items()}
    A = torch.from_numpy(inp.A).to(dev)
    Dk = torch.from_numpy(inp.D).to(dev)
    init = None if inp.init is None else torch.from_numpy(inp.init).to(dev)
    b, L, D, N = shape["batch"], shape["seqlen"], shape["dim"], shape["dstate"]
    y = torch.empty_like(d["x"])
    fin = torch.empty((b, D, N), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(k):
        flush.fill_(k & 0xFF)
        flush_rd.max()

    def step():
        ssd.selective_scan(d["x"], d["delta"], A, d["B"], d["C"], Dk, init, y=y, final_state=fin,
                           stream=stream)

    for k in range(max(3, args.warmup)):
        flush_l2(k)
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for k in range(args.steps):
        flush_l2(k)
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    ms_step = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    ms_step = max_over_ranks(ms_step, ws, dist, dev)
    tokens = b * L
    value = job_rate(tokens, ws, ms_step)
    e = 2 if bf16 else 4
    elems = b * L * D * N
    hbm_bytes = 3 * b * L * D * e + 2 * b * L * N * e + D * N * 4 + D * 4 + (2 if init is not None else 1) * b * D * N * 4
    ach = elems / (ms_step * 1e-3) / 1e9
    roofline = {"kernel": "selective_scan", "bound": "alu", "achieved": ach, "peak": MUFU_PEAK_GPS,
                "unit": "Gexp/s", "frac": ach / MUFU_PEAK_GPS, "traffic": profiled_traffic("selective_scan", args.workload),
                "peak_source": "derived: 152 SMs x 32 MUFU ex2 per clock x 2.07 GHz (one exp per element)",
                "hbm_context": {"bytes": hbm_bytes, "GBps": hbm_bytes / (ms_step * 1e-3) / 1e9}}

    e2e = None
    if not args.no_e2e:
        pin = {k: v.pin_memory() for k, v in host.items()}
        ys = [y, torch.empty_like(y)]
        fins = [fin, None if fin is None else torch.empty_like(fin)]

        def sel_slot(src, i):
            yy, _ = ssd.selective_scan(src["x"], src["delta"], A, src["B"], src["C"], Dk, init,
                                       y=ys[i], final_state=fins[i])
            return [yy]

        ms_e2e, h2d, d2h = pipelined_e2e(torch, dev, args.steps, pin, sel_slot)
        ms_e2e = max_over_ranks(ms_e2e, ws, dist, dev)
        e2e = {"value": job_rate(tokens, ws, ms_e2e), "unit": "tokens/s", "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipelined": "upload / compute / download streams, two buffer sets"}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline_selective(inp, args.cpu_seconds)
    line = {
        "metric": METRIC_SEL, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16 else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": args.workload, **shape,
                   "l2": "flushed before every step (256 MiB write + 256 MiB read, outside the timed events)",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": roofline,
        "kernels": {"selective_scan": {"us": 1e3 * ms_step, "share": 1.0, "elements": elems,
                                        "hbm_bytes": hbm_bytes}},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_decode(args, torch, dist, ssd, ws, rank, local, dev, shape, inp, host, d):
    """The decode arm: one ssd_decode launch per step over resident state and inputs."""
    b, T, H, P, N = (shape[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate"))
    state = (d["init"].clone() if d["init"] is not None
             else torch.zeros((b, H, P, N), dtype=torch.float32, device=dev))
    y = torch.empty_like(d["x"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(k):
        flush.fill_(k & 0xFF)
        flush_rd.max()

    def step():
        ssd.decode(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], state, y=y, stream=stream)

    for k in range(max(3, args.warmup)):
        flush_l2(k)
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for k in range(args.steps):
        flush_l2(k)
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    ms_step = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    ms_step = max_over_ranks(ms_step, ws, dist, dev)
    tokens = b * T
    value = job_rate(tokens, ws, ms_step)
    by, fl = algorithmic_decode(shape)
    peaks = load_peaks()
    ach = by / (ms_step * 1e-3) / 1e9
    roofline = {"kernel": "decode", "bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": ach / peaks["hbm"], "traffic": profiled_traffic("decode", args.workload),
                "peak_source": peaks["src"] + " (MEASURED_PEAKS.json burst)"
                if peaks["src"] == "measured" else "fallback"}

    # end to end: the step's token inputs (x, dt, B, C) from pinned host memory, y back to pinned
    # host memory; the state stays resident on the device (it is the cache being decoded from)
    e2e = None
    if not args.no_e2e:
        # one stream: a decode step moves about a megabyte, too little for the upload / compute /
        # download pipeline of the other workloads to pay for its extra synchronisation
        pin = {k: host[k].pin_memory() for k in ("x", "dt", "B", "C")}
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        dev_in = {k: torch.empty_like(v, device=dev) for k, v in pin.items()}
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = y_host.numel() * y_host.element_size()

        def e2e_step():
            for k, v in pin.items():
                dev_in[k].copy_(v, non_blocking=True)
            yy = ssd.decode(dev_in["x"], dev_in["dt"], d["A"], dev_in["B"], dev_in["C"], d["D"], state,
                            y=y, stream=stream)
            y_host.copy_(yy, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = e0.elapsed_time(e1) / args.steps
        ms_e2e = max_over_ranks(ms_e2e, ws, dist, dev)
        e2e = {"value": job_rate(tokens, ws, ms_e2e), "unit": "tokens/s", "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "note": "state resident on the device across steps"}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline(inp, args.cpu_seconds)
    line = {
        "metric": METRIC_DECODE, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if inp.io_dtype == "bf16" else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": args.workload, **shape,
                   "l2": "flushed before every step (256 MiB write + 256 MiB read, outside the timed events)",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "state": "float32 (b, H, P, N), read and written once per step"},
        "roofline": roofline,
        "kernels": {"decode": {"us": 1e3 * ms_step, "share": 1.0, "alg_bytes": by, "alg_flops": fl}},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
