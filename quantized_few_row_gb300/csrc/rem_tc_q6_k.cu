// Instantiates rem_tc_kernel<kQ6_K, MP, CM> for the tile widths MP = 1, 2, 4, 8, 16.
#include "rem_tc.cuh"

REM_TC_INSTANTIATE(rem::kQ6_K, tc_kernel_q6_k)
