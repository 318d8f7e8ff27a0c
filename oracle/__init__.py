"""TEST INFRASTRUCTURE -- the double-precision CPU oracles of the mHC pre forward,
its backward, and the post-mapping (hc_post).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never does, and this package never imports the product.

``build()`` compiles ``mhc_pre_oracle.c``, ``mhc_pre_bwd_oracle.c`` and
``mhc_post_oracle.c`` with gcc into ``_build/`` next to this file; ``run()``,
``run_backward()`` and ``run_post()`` call them through ctypes on numpy arrays
and return the outputs in float64.
"""
from .oracle import (build, run, run_backward, run_post, half_value, OracleOut, BwdOut,  # noqa: F401
                     brute_force_decimal)
