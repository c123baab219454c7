// Fused layer kernels for K = 5 bits per weight (one translation unit per K so
// the library builds in parallel).
#include "exl3_layer.cuh"
EXL3_DEFINE_LAYER_LAUNCHER(5)
