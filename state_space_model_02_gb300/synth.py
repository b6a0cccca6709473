"""Seeded synthetic inputs for the SSD forward scan (shared by tests, bench, oracle checks).

This module draws random numbers and rounds them to the I/O dtype; it holds
none of the layer's arithmetic.  One ``numpy.random.default_rng(seed)`` stream
is drawn in the fixed order x, B, C, dt_raw, A_u, D, init, so the GPU path and
the CPU oracle see bit-identical inputs.

Distributions (the workloads of "Mamba-2 cuda-tile forward pass kernels",
section 4: 1K-256K tokens, state sizes 64-512, chunk 256; Mamba-2 130M / 2.7B
layer shapes):
  x, B, C ~ N(0, 1), rounded to bf16 (round-to-nearest-even) or kept fp32
  dt      = clip(softplus(N(-3, 1)), 1e-3, 0.1)            float32
  A       = -exp(U(ln a_lo, ln a_hi)), default [-16, -1]   float32
  D       ~ N(0, 1)                                        float32
  init    ~ N(0, 0.1) when requested, else absent          float32
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# Workloads: name -> shape.  chunk is the SSD chunk length Q.
CONFIGS = {
    "tiny_fp32": dict(batch=1, seqlen=256, nheads=4, headdim=16, dstate=16, ngroups=1, chunk=64,
                      io_dtype="f32", init=False),
    "mamba2_130m_layer": dict(batch=4, seqlen=2048, nheads=24, headdim=64, dstate=128, ngroups=1,
                              chunk=256, io_dtype="bf16", init=False),
    "mamba2_2p7b_layer": dict(batch=2, seqlen=8192, nheads=80, headdim=64, dstate=128, ngroups=1,
                              chunk=256, io_dtype="bf16", init=True),
    "state_sweep_n64": dict(batch=1, seqlen=16384, nheads=32, headdim=64, dstate=64, ngroups=1,
                            chunk=256, io_dtype="bf16", init=False),
    "state_sweep_n128": dict(batch=1, seqlen=16384, nheads=32, headdim=64, dstate=128, ngroups=1,
                             chunk=256, io_dtype="bf16", init=False),
    "state_sweep_n256": dict(batch=1, seqlen=16384, nheads=32, headdim=64, dstate=256, ngroups=1,
                             chunk=256, io_dtype="bf16", init=False),
    "state_sweep_n512": dict(batch=1, seqlen=16384, nheads=32, headdim=64, dstate=512, ngroups=1,
                             chunk=256, io_dtype="bf16", init=False),
    "long_256k": dict(batch=1, seqlen=262144, nheads=32, headdim=64, dstate=128, ngroups=1,
                      chunk=256, io_dtype="bf16", init=False),
    # decoding (the recurrent form): seqlen is the number of tokens one launch advances the
    # state by; the state (b, H, P, N) float32 is the whole per-sequence cache
    "decode_2p7b_b64_t1": dict(batch=64, seqlen=1, nheads=80, headdim=64, dstate=128, ngroups=1,
                               chunk=64, io_dtype="bf16", init=True),
    "decode_2p7b_b64_t16": dict(batch=64, seqlen=16, nheads=80, headdim=64, dstate=128, ngroups=1,
                                chunk=64, io_dtype="bf16", init=True),
}


@dataclass
class SSDInputs:
    """Host arrays of one problem.  x/B/C: float32, or uint16 holding bf16 bits."""
    x: np.ndarray
    dt: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    D: Optional[np.ndarray]
    init: Optional[np.ndarray]
    chunk: int
    io_dtype: str
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        b, L, H, P = self.x.shape
        return dict(batch=b, seqlen=L, nheads=H, headdim=P, dstate=self.B.shape[3],
                    ngroups=self.B.shape[2], chunk=self.chunk, io_dtype=self.io_dtype)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32, exactly."""
    return (np.asarray(a, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_inputs(batch, seqlen, nheads, headdim, dstate, ngroups=1, chunk=256, io_dtype="bf16",
                init=False, seed=0, a_range=(1.0, 16.0), with_D=True, dt_mean=-3.0,
                dt_clip=(1e-3, 0.1)) -> SSDInputs:
    """Draw one problem from the distributions in the module docstring.

    dt_mean and dt_clip move the step-size distribution (softplus(N(dt_mean, 1)) clipped to
    dt_clip) for the large-step edge cases; the defaults are the workloads' recipe."""
    if io_dtype not in ("bf16", "f32"):
        raise ValueError("io_dtype must be 'bf16' or 'f32'")
    rng = np.random.default_rng(seed)
    b, L, H, P, N, G = batch, seqlen, nheads, headdim, dstate, ngroups
    x = rng.standard_normal((b, L, H, P), dtype=np.float32)
    Bm = rng.standard_normal((b, L, G, N), dtype=np.float32)
    Cm = rng.standard_normal((b, L, G, N), dtype=np.float32)
    dt_raw = rng.normal(dt_mean, 1.0, size=(b, L, H))
    a_u = rng.uniform(np.log(a_range[0]), np.log(a_range[1]), size=H)
    D = rng.standard_normal(H).astype(np.float32)
    h0 = rng.normal(0.0, 0.1, size=(b, H, P, N)).astype(np.float32) if init else None
    dt = np.clip(np.logaddexp(0.0, dt_raw), dt_clip[0], dt_clip[1]).astype(np.float32)
    A = (-np.exp(a_u)).astype(np.float32)
    if io_dtype == "bf16":
        x, Bm, Cm = to_bf16_bits(x), to_bf16_bits(Bm), to_bf16_bits(Cm)
    return SSDInputs(x=x, dt=dt, A=A, B=Bm, C=Cm, D=D if with_D else None, init=h0, chunk=chunk,
                     io_dtype=io_dtype, meta=dict(seed=seed, a_range=tuple(a_range), dt_mean=dt_mean,
                                                  dt_clip=tuple(dt_clip)))


def make_config(name: str, seed: int = 0, **overrides) -> SSDInputs:
    """Inputs of a named workload from CONFIGS (overrides patch the shape)."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    return make_inputs(seed=seed, **cfg)


# ---------------------------------------------------------------- Mamba-1 selective scan
#
# "3.3 Hardware-aware algorithm and GPU memory hierarchy", section 2.1: x and delta are
# (batch, L, D) with D channels, B and C (batch, L, N), A one value per (channel, state).
# Layer shapes of Mamba-1 130M / 2.8B (d_inner 1536 / 5120, state 16); section 5.1's
# sequences of 8192 tokens and more.  Same distributions as above, drawn in the order
# x, B, C, delta_raw, A_u, D, init:
#   x, B, C ~ N(0, 1) in the I/O dtype; delta = clip(softplus(N(-3, 1)), 1e-3, 0.1) in the
#   I/O dtype; A (D, N) = -exp(U(ln a_lo, ln a_hi)); Dskip ~ N(0, 1); init (b, D, N) ~ N(0, 0.1).

SELECTIVE_CONFIGS = {
    "mamba1_tiny_fp32": dict(batch=1, seqlen=256, dim=64, dstate=16, io_dtype="f32", init=False),
    "mamba1_130m_layer": dict(batch=4, seqlen=2048, dim=1536, dstate=16, io_dtype="bf16", init=False),
    "mamba1_2p8b_layer": dict(batch=2, seqlen=8192, dim=5120, dstate=16, io_dtype="bf16", init=True),
}


@dataclass
class SelectiveInputs:
    """Host arrays of one selective-scan problem.  x/delta/B/C: float32 or bf16 bits (uint16)."""
    x: np.ndarray
    delta: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    D: Optional[np.ndarray]
    init: Optional[np.ndarray]
    io_dtype: str
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        b, L, D = self.x.shape
        return dict(batch=b, seqlen=L, dim=D, dstate=self.B.shape[2], io_dtype=self.io_dtype)


def make_selective_inputs(batch, seqlen, dim, dstate, io_dtype="bf16", init=False, seed=0,
                          a_range=(1.0, 16.0), with_D=True) -> SelectiveInputs:
    if io_dtype not in ("bf16", "f32"):
        raise ValueError("io_dtype must be 'bf16' or 'f32'")
    rng = np.random.default_rng(seed)
    b, L, D, N = batch, seqlen, dim, dstate
    x = rng.standard_normal((b, L, D), dtype=np.float32)
    Bm = rng.standard_normal((b, L, N), dtype=np.float32)
    Cm = rng.standard_normal((b, L, N), dtype=np.float32)
    d_raw = rng.normal(-3.0, 1.0, size=(b, L, D))
    a_u = rng.uniform(np.log(a_range[0]), np.log(a_range[1]), size=(D, N))
    Dskip = rng.standard_normal(D).astype(np.float32)
    h0 = rng.normal(0.0, 0.1, size=(b, D, N)).astype(np.float32) if init else None
    delta = np.clip(np.logaddexp(0.0, d_raw), 1e-3, 0.1).astype(np.float32)
    A = (-np.exp(a_u)).astype(np.float32)
    if io_dtype == "bf16":
        x, Bm, Cm, delta = to_bf16_bits(x), to_bf16_bits(Bm), to_bf16_bits(Cm), to_bf16_bits(delta)
    return SelectiveInputs(x=x, delta=delta, A=A, B=Bm, C=Cm, D=Dskip if with_D else None, init=h0,
                           io_dtype=io_dtype, meta=dict(seed=seed, a_range=tuple(a_range)))


def make_selective_config(name: str, seed: int = 0, **overrides) -> SelectiveInputs:
    cfg = dict(SELECTIVE_CONFIGS[name])
    cfg.update(overrides)
    return make_selective_inputs(seed=seed, **cfg)
