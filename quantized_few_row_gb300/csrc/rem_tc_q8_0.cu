// Instantiates rem_tc_kernel<kQ8_0, MP> for MP = 8, 16, 32.
#include "rem_tc.cuh"

REM_TC_INSTANTIATE(rem::kQ8_0, tc_kernel_q8_0)
