"""GB300 (sm_103a) Mamba-2 SSD chunked forward scan.

The work runs in libssd.so (hand-written CUDA: chunk_cumsum, chunk_state,
state_passing, chunk_scan) behind the C ABI in include/ssd.h; ``ssd`` is the
ctypes binding and ``synth`` the seeded input generator.
"""
from . import ssd  # noqa: F401
from .ssd import fwd, workspace_bytes, Problem, SSDError  # noqa: F401
