"""Oracle for the shared-memory-operand GEMM: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(``cpu_baseline`` / ``--impl reference``) may import, call or link anything in
this package.  The product path (the CUDA library and its Python binding) never
does, and shares no code with it.

Contents
  gemm.py     fp64 CPU GEMM (plain C through ctypes) + exact rational brute
              force; IEEE round-to-nearest-even to f32 / bf16 / f16.
  f2.py       linear layouts over F2 (apply, invert, invert-and-compose,
              left division) as the MI450 LDS post defines them.
  banksim.py  bank-conflict simulator (banks, phases, broadcast) and the GB300
              128-byte-swizzled tile layouts restated from their definitions.

Pins (tests/test_oracle_*.py, marked "not gpu") tie each function to values the
pages print or to the mathematics: exact brute force, identity / permutation /
closed-form products, library cross-checks, the pages' worked tables.
"""
