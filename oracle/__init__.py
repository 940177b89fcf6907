"""CPU oracle for the TurboQuant KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) may
import anything from this package.  The product path -- the CUDA library under
``kv_cache_quantization_random_gb300/`` and its Python binding -- never imports
it, and the two share no code, tables or constants: each derives the codebook,
the sign vectors and the QJL matrix on its own from the published definitions.

Everything here is plain fp64 NumPy (and the ``math`` module), written for a
reader to check against the pages by eye, not for speed.

Parity status of each function is stated in its docstring; the pins live in
``tests/test_oracle_pins.py``.  The whole pipeline is pinned piecewise; the
exact constants of the seeded generators (splitmix64 streams, Box-Muller) have
no external reference beyond the published splitmix64 test values, so the
*choice* of stream layout is a convention both sides implement independently.
"""

from .tq_oracle import *  # noqa: F401,F403
