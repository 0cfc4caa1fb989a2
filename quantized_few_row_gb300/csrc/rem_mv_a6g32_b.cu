// Instantiates rem_mv_kernel<kA6G32, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kA6G32, mv_kernel_a6g32_b, 5, 4)
