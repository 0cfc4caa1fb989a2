// Instantiates rem_mv_kernel<kQ5_0, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kQ5_0, mv_kernel_q5_0_b, 5, 4)
