// Instantiates rem_mv_kernel<kA3G128, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kA3G128, mv_kernel_a3g128_a, 1, 4)
