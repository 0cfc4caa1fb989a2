// Instantiates rem_mv_kernel<kQ8_0, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kQ8_0, mv_kernel_q8_0_b, 5, 4)
