// Instantiates rem_mv_kernel<kF16, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kF16, mv_kernel_f16_b, 5, 4)
