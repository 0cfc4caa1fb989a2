// Instantiates rem_mv_kernel<kQ5_0, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kQ5_0, mv_kernel_q5_0_a, 1, 4)
