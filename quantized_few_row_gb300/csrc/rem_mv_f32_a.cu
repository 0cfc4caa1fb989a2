// Instantiates rem_mv_kernel<kF32, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kF32, mv_kernel_f32_a, 1, 4)
