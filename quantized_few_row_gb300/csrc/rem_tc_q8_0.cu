// Instantiates rem_tc_kernel<kQ8_0, MP, CM> for the tile widths MP = 1, 2, 4, 8, 16, 32.
#include "rem_tc.cuh"

REM_TC_INSTANTIATE(rem::kQ8_0, tc_kernel_q8_0)
