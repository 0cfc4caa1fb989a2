// Instantiates rem_mv_kernel<kA6G32, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kA6G32, mv_kernel_a6g32_a, 1, 4)
