// Instantiates rem_mv_kernel<kA5G64, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kA5G64, mv_kernel_a5g64_a, 1, 4)
