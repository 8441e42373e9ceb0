"""CPU oracle for the stream-K GEMM / implicit-GEMM conv wgrad / fp8 row-col GEMM path.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, call, link or run anything
in this package. The CUDA path never calls it and shares no code with it.

Contents:

* ``codec``     -- binary16 / bfloat16 / OCP E4M3 decode and round-to-nearest-even encode.
* ``partition`` -- the stream-K iteration partitioner restated step by step, a brute-force
                   iteration assignment, the partition invariants and a forward-progress simulator.
* ``ref.c``     -- fp64 GEMM (rcr), direct-loop NHWC wgrad and fp8 row/col-scaled GEMM (plain C,
                   OpenMP over independent outputs), loaded through ``oracle.numerics``.

Every function is pinned by ``tests/test_oracle_*.py`` against something other than itself
(library routines in fp64, closed forms, exhaustive format tables, brute force).
"""
