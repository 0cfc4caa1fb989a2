// Instantiates rem_mv_kernel<kF32, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kF32, mv_kernel_f32_b, 5, 4)
