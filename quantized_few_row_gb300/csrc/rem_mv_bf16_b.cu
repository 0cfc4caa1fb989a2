// Instantiates rem_mv_kernel<kBF16, M, NR0, H> for M = 5..8.
#include "rem_mv.cuh"

REM_INSTANTIATE(rem::kBF16, mv_kernel_bf16_b, 5, 4)
