// Host-side helpers of libexl3: argument validation, launch plans and the
// internal launcher declarations shared by the translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/exl3.h"

namespace exl3 {

constexpr int kRowBlock = 128;      // rows per output block (one output FWHT)
constexpr int kMaxSplits = 64;      // cap on K-dimension slices of one layer
constexpr size_t kXsBudget = 96 * 1024;  // smem bytes for the rotated x slice

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline exl3_status check_shape(int m, int n) {
  if (m <= 0 || n <= 0 || (m % kRowBlock) != 0 || (n % kRowBlock) != 0) return EXL3_ERR_SHAPE;
  return EXL3_OK;
}

inline exl3_status check_k_cb(int K, int codebook) {
  if (K < 1 || K > 8) return EXL3_ERR_K;
  if (codebook != EXL3_CB_3INST && codebook != EXL3_CB_1MAD) return EXL3_ERR_CODEBOOK;
  return EXL3_OK;
}

inline exl3_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? EXL3_OK : EXL3_ERR_CUDA;
}

// Number of SMs of the current device (queried once per device).
int device_sm_count();

// Workspace layout: [counters: one uint32 per 128-row block, then one status
// word (non-zero after a device-side wait timed out), padded to 256 B]
// [partials: fp32 [splits][M][m]].
inline size_t counters_bytes(int m) {
  const size_t b = sizeof(uint32_t) * (static_cast<size_t>(m / kRowBlock) + 1);
  return (b + 255) & ~static_cast<size_t>(255);
}
inline int max_splits(int n) {
  const int nblk = n / kRowBlock;
  return nblk < kMaxSplits ? nblk : kMaxSplits;
}

// Split count of the K dimension for an m x n layer at batch chunk mb: enough
// CTAs to cover every SM a few times, each slice a whole number of 128-column
// blocks, and the rotated x slice within the shared-memory budget.
int choose_splits(int m, int n, int mb, int sm_count);

struct LayerArgs {
  const uint32_t* codes;
  int K, codebook, m, n;
  const __half* s_in;
  const __half* s_out;
  const __half* scales;
  const __half* x;  // [mb][n]
  __half* y;        // [mb][m]
  float* partials;
  uint32_t* counters;
  uint32_t* status;  // device-side error bits (tensor-core path), or nullptr
  int splits;
};

// Internal launchers (one translation unit per K for the layer kernels).
exl3_status launch_rht(const __half* in, const __half* signs, __half* out, int rows, int d,
                       cudaStream_t stream);
exl3_status launch_decode(const uint32_t* codes, int K, int codebook, int m, int n, __half* w,
                          cudaStream_t stream);
exl3_status launch_layer_k1(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k2(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k3(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k4(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k5(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k6(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k7(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k8(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_tc_k1(const LayerArgs& a, int M, cudaStream_t stream);
exl3_status launch_tc_k2(const LayerArgs& a, int M, cudaStream_t stream);
exl3_status launch_tc_k3(const LayerArgs& a, int M, cudaStream_t stream);
exl3_status launch_tc_k4(const LayerArgs& a, int M, cudaStream_t stream);
exl3_status launch_tc_k5(const LayerArgs& a, int M, cudaStream_t stream);
exl3_status launch_tc_k6(const LayerArgs& a, int M, cudaStream_t stream);
exl3_status launch_tc_k7(const LayerArgs& a, int M, cudaStream_t stream);
exl3_status launch_tc_k8(const LayerArgs& a, int M, cudaStream_t stream);

// Split count for the tensor-core path: about two resident CTAs per SM, and
// slices of at most kTcMaxSliceCols columns (the duplicated x slice lives in
// shared memory).
constexpr int kTcMaxSliceCols = 1024;
int choose_tc_splits(int m, int n, int sm_count);

}  // namespace exl3
