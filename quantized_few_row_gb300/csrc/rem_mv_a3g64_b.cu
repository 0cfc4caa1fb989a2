// Instantiates rem_mv_kernel<kA3G64, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kA3G64, mv_kernel_a3g64_b, 5, 4)
