"""CPU oracle for the fp16 GEMM with fp32 accumulation and the grouped tile map.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (and its ``--impl reference`` arm) may import,
call, link or execute anything in this package. The product library
(``dense_fp16_gemm_fp32_gb300``) never does; the two share no code.

Contents:
  tile_map.py      the grouped program-id -> (pid_m, pid_n) map, pure ints
  gemm_oracle.c    the GEMM oracle, plain C: fp32 sum in ascending k, one
                   round-to-nearest-even narrowing to fp16
  gemm.py          ctypes front end of gemm_oracle.c
  build.py         gcc build of gemm_oracle.c
  softmax.py       the row softmax of the fused-softmax tutorial, numpy fp64

Pins (the tests that tie the oracle to something other than itself):
  tile map         the notebook's printed worked example (tests/golden/),
                   bijection sweeps, the closed forms for GROUP_SIZE_M == 1
                   and GROUP_SIZE_M >= num_pid_m, an independent nested-loop
                   construction for every unclamped group, and the
                   notebook's printed pointer matrices for program 60.
  fp16 conversion  exhaustive comparison with numpy/torch conversions.
  GEMM             fp64 brute force within the recursive-summation bound,
                   identity and zero matrices, exact small-integer products,
                   order-sensitive sums whose ascending-k fp32 value is known
                   in closed form, and the single-narrowing case.
No function here is "parity unpinned".
"""
