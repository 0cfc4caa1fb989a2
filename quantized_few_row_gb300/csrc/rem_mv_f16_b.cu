// Instantiates rem_mv_kernel<kF16, M, NR0> for M = 5..8 and NR0 = 1, 2.
#include "rem_mv.cuh"

REM_INSTANTIATE4(rem::kF16, mv_kernel_f16_b, 5)
