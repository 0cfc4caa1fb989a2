// Instantiates rem_mv_kernel<kQ6_K, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kQ6_K, mv_kernel_q6_k_a, 1, 4)
