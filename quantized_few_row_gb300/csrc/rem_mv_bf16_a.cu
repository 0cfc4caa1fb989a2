// Instantiates rem_mv_kernel<kBF16, M, NR0, H> for M = 1..4.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kBF16, mv_kernel_bf16_a, 1, 4)
