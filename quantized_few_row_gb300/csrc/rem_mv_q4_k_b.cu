// Instantiates rem_mv_kernel<kQ4_K, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kQ4_K, mv_kernel_q4_k_b, 5, 4)
