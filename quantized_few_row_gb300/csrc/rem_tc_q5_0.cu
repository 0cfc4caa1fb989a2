// Instantiates rem_tc_kernel<kQ5_0, MP> for MP = 8, 16, 32.
#include "rem_tc.cuh"

REM_TC_INSTANTIATE(rem::kQ5_0, tc_kernel_q5_0)
