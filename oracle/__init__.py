"""CPU oracle for the Mamba-2 SSD chunked forward scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import anything from this package.  The GPU product
path (``state_space_model_02_gb300``) shares no code with it and never calls it.

Contents
--------
ssd_ref.c      float64 token-by-token recurrence (the definition), OpenMP over
               (batch, head) pairs; also per-chunk zero-start end states.
ref.py         ctypes front end for ssd_ref.c plus NumPy float64 forms that pin
               it: the quadratic (dual) form, an independent chunked evaluation,
               the in-chunk log2 cumsum, and closed forms for special cases.
build.py       compiles ssd_ref.c with gcc (no GPU, no CUDA).

Every function states the passage it follows.  Nothing here is "parity
unpinned": each function has at least one test in ``tests/test_oracle_*.py``
that checks it against something other than itself.
"""
