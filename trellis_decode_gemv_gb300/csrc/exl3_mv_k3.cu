// Decode-MMA layer kernel (codes decoded into tensor memory, tcgen05 MMAs,
// input and output transforms in the same launch) for K = 3 bits per weight,
// one translation unit per K.
#include "exl3_mv.cuh"
EXL3_DEFINE_MV_LAUNCHER(3)
