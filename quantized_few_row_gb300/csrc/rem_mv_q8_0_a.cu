// Instantiates rem_mv_kernel<kQ8_0, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kQ8_0, mv_kernel_q8_0_a, 1, 4)
