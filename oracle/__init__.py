"""TEST INFRASTRUCTURE -- the double-precision CPU oracle of the mHC pre forward.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never does, and this package never imports the product.

``build()`` compiles ``mhc_pre_oracle.c`` with gcc into ``_build/`` next to
this file; ``run()`` calls it through ctypes on numpy arrays and returns the
outputs in float64.
"""
from .oracle import build, run, OracleOut, brute_force_decimal  # noqa: F401
