// Fused layer kernels, binary16 and int8 activations, for K = 3 bits per
// weight (one translation unit per K so the library builds in parallel).
#include "exl3_layer.cuh"
#include "exl3_i8.cuh"
EXL3_DEFINE_LAYER_LAUNCHER(3)
EXL3_DEFINE_I8_LAUNCHER(3)
