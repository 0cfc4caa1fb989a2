// Instantiates rem_mv_kernel<kQ6_K, M, NR0> for M = 1..4 and NR0 = 1, 2.
#include "rem_mv.cuh"

REM_INSTANTIATE4(rem::kQ6_K, mv_kernel_q6_k_a, 1)
