// Instantiates rem_mv_kernel<kF16, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kF16, mv_kernel_f16_a, 1, 4)
