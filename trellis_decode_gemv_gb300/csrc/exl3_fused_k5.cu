// Fused prefill kernel (codes decoded into operand A in shared memory, then
// tcgen05 MMAs) for K = 5 bits per weight, one translation unit per K.
#include "exl3_dense.cuh"
EXL3_DEFINE_FUSED_LAUNCHER(5)
