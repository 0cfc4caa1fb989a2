// Instantiates rem_mv_kernel<kA3G32, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kA3G32, mv_kernel_a3g32_b, 5, 4)
