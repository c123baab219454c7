// Tensor-core fused layer kernels for K = 6 bits per weight.
#include "exl3_tc.cuh"
EXL3_DEFINE_TC_LAUNCHER(6)
