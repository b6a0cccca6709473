"""Shared helpers for the tests: device copies of synthetic inputs and oracle comparisons."""
import numpy as np

from oracle import ref
from state_space_model_02_gb300 import synth

TOL = {"bf16": 2e-2, "f32": 1e-4}


def to_device(inp, device="cuda"):
    """Device tensors (x, dt, A, B, C, D, init) of an SSDInputs, bit-identical to the host arrays."""
    import torch

    bf16 = inp.io_dtype == "bf16"

    def io(a):
        if bf16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    def f32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)

    return dict(x=io(inp.x), dt=f32(inp.dt), A=f32(inp.A), B=io(inp.B), C=io(inp.C), D=f32(inp.D),
                init=f32(inp.init))


def y_to_numpy(y):
    import torch

    return y.float().cpu().numpy() if y.dtype == torch.bfloat16 else y.cpu().numpy()


def oracle_pairs(inp, pairs, want_chunk_in=False):
    """Oracle recurrence for selected (b, h) pairs; y as (nsel, L, P)."""
    return ref.recurrence(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.init, chunk=inp.chunk,
                          pairs=np.asarray(pairs, np.int64), want_chunk_in=want_chunk_in)


def sample_pairs(batch, nheads, k, seed=0):
    """k distinct (b, h) pairs, always including the first and the last."""
    rng = np.random.default_rng(seed)
    allp = [(b, h) for b in range(batch) for h in range(nheads)]
    if k >= len(allp):
        return allp
    idx = set(rng.choice(len(allp), size=k - 2, replace=False).tolist()) | {0, len(allp) - 1}
    return [allp[i] for i in sorted(idx)]


def gather_y(y_np, pairs):
    """(nsel, L, P) slices of a (b, L, H, P) array for the given pairs."""
    return np.stack([y_np[b, :, h, :] for b, h in pairs])


def rel(got, want):
    return ref.rel_err(got, want)


def make(name_or_shape, **kw):
    if isinstance(name_or_shape, str):
        return synth.make_config(name_or_shape, **kw)
    return synth.make_inputs(**name_or_shape, **kw)
