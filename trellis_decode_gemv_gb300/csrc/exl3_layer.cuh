// Fused layer kernel, warp-shuffle path:
//   y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x))))
// ("ExLlamaV3 & EXL3 Deep Dive" Section 2 runtime identity; W-hat decoded on
// the fly from the bitshift-trellis codes of "Trellis Quantization" Parts
// eight and nine; blockwise 128-point transforms of Part eleven).
//
// One CTA = one 128-row output block x one slice of the input dimension
// (a whole number of 128-column blocks).  8 warps, warp w owns tile-row
// 8*blockIdx.x + w.  Inside a warp, lane = 8*jt + p: jt picks every 4th tile
// of the slice, p the row pair (rows 2p, 2p+1) of the tile, so each thread
// decodes 32 consecutive trellis steps from a word-aligned window.
//
// Prologue: the slice of x is rotated (signs, 128-point FWHT across a warp,
// 1/sqrt(128)) into shared memory as fp32, times the code's x factor (see
// decode_f32).  Main loop: all 32 trellis states of a row pair, decode to fp32,
// FMA into two row accumulators per batch row, with the next tile's words
// loaded before the current tile is decoded.  Then a warp-shuffle reduction over the
// 4 tile groups, and, when the input dimension is split, a last-arriving-CTA
// combine (fp32 partials in the workspace + one atomic ticket per row block;
// no CTA ever waits on another).  Epilogue: scale, output signs, 128-point
// FWHT across a warp, binary16 store.
#pragma once

#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {

constexpr int kLayerThreads = 256;

__device__ __forceinline__ void load_half4(const __half* p, float (&v)[4]) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  const __half2 a = *reinterpret_cast<const __half2*>(&r.x);
  const __half2 b = *reinterpret_cast<const __half2*>(&r.y);
  v[0] = __low2float(a);
  v[1] = __high2float(a);
  v[2] = __low2float(b);
  v[3] = __high2float(b);
}

__device__ __forceinline__ void store_half4(__half* p, const float (&v)[4]) {
  const __half2 a = __floats2half2_rn(v[0], v[1]);
  const __half2 b = __floats2half2_rn(v[2], v[3]);
  uint2 r;
  r.x = *reinterpret_cast<const uint32_t*>(&a);
  r.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = r;
}

template <int K, int CB, int MB>
__global__ void __launch_bounds__(kLayerThreads) layer_kernel(LayerArgs a) {
  extern __shared__ __align__(16) float smem[];
  __shared__ uint32_t s_ticket;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int rb = blockIdx.x;
  const int split = blockIdx.y;
  const int nblk = a.n / kRowBlock;
  const int kb0 = static_cast<int>(static_cast<long long>(split) * nblk / a.splits);
  const int kb1 = static_cast<int>(static_cast<long long>(split + 1) * nblk / a.splits);
  const int c0 = kb0 * kRowBlock;
  const int ns = (kb1 - kb0) * kRowBlock;
  float* xs = smem;            // [MB][ns] rotated x slice
  float* zs = smem + MB * ns;  // [MB][128] row sums of this block

  // ---- prologue: rotate the x slice into shared memory -------------------
  const int nkb = ns / kRowBlock;
  for (int job = warp; job < MB * nkb; job += kLayerThreads / 32) {
    const int b = job / nkb;
    const int kb = job - b * nkb;
    const int col = c0 + kb * kRowBlock + 4 * lane;
    float v[4];
    load_half4(a.x + static_cast<size_t>(b) * a.n + col, v);
    if (a.s_in != nullptr) {
      float s[4];
      load_half4(a.s_in + col, s);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] *= s[j];
      fwht128_warp(v, lane);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] *= x_factor<CB>();
    *reinterpret_cast<float4*>(xs + b * ns + kb * kRowBlock + 4 * lane) =
        make_float4(v[0], v[1], v[2], v[3]);
  }
  __syncthreads();

  // ---- main loop: decode + fp32 FMA ---------------------------------------
  constexpr int kTw = RowPair<K>::kTileWords;
  const int I = rb * (kRowBlock / 16) + warp;
  const int jt = lane >> 3;
  const int p = lane & 7;
  const int tiles_per_row = a.n / 16;
  const uint32_t* rowp = a.codes + static_cast<size_t>(I) * tiles_per_row * kTw;
  float acc[MB][2];
#pragma unroll
  for (int b = 0; b < MB; ++b) acc[b][0] = acc[b][1] = 0.f;

  const int J0 = c0 / 16;
  const int J1 = (c0 + ns) / 16;
  int J = J0 + jt;
  uint32_t w[RowPair<K>::kPairWords];
  if (J < J1) load_row_pair<K>(rowp + static_cast<size_t>(J) * kTw, p, w);
  while (J < J1) {
    uint32_t st[32];
    pair_states<K>(w, st);
    const int Jc = J;
    J += 4;
    if (J < J1) load_row_pair<K>(rowp + static_cast<size_t>(J) * kTw, p, w);  // prefetch
    const float* xt = xs + (Jc * 16 - c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float wa[4], wb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wa[j] = decode_f32<CB>(st[4 * q + j]);
        wb[j] = decode_f32<CB>(st[16 + 4 * q + j]);
      }
#pragma unroll
      for (int b = 0; b < MB; ++b) {
        const float4 xv = *reinterpret_cast<const float4*>(xt + b * ns + 4 * q);
        acc[b][0] = fmaf(wa[0], xv.x, acc[b][0]);
        acc[b][0] = fmaf(wa[1], xv.y, acc[b][0]);
        acc[b][0] = fmaf(wa[2], xv.z, acc[b][0]);
        acc[b][0] = fmaf(wa[3], xv.w, acc[b][0]);
        acc[b][1] = fmaf(wb[0], xv.x, acc[b][1]);
        acc[b][1] = fmaf(wb[1], xv.y, acc[b][1]);
        acc[b][1] = fmaf(wb[2], xv.z, acc[b][1]);
        acc[b][1] = fmaf(wb[3], xv.w, acc[b][1]);
      }
    }
  }

  // ---- warp-shuffle reduction over the 4 tile groups -----------------------
#pragma unroll
  for (int b = 0; b < MB; ++b) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float v = acc[b][k];
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
      acc[b][k] = v;
    }
  }
  if (jt == 0) {
#pragma unroll
    for (int b = 0; b < MB; ++b) {
      zs[b * kRowBlock + warp * 16 + 2 * p] = acc[b][0];
      zs[b * kRowBlock + warp * 16 + 2 * p + 1] = acc[b][1];
    }
  }
  __syncthreads();

  // ---- split-K combine: the last CTA of this row block sums the partials ---
  if (a.splits > 1) {
    float* part = a.partials + static_cast<size_t>(split) * MB * a.m;
    for (int i = tid; i < MB * kRowBlock; i += kLayerThreads) {
      const int b = i / kRowBlock;
      const int r = i - b * kRowBlock;
      part[static_cast<size_t>(b) * a.m + rb * kRowBlock + r] = zs[i];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_ticket = atomicAdd(a.counters + rb, 1u);
    __syncthreads();
    if (s_ticket != static_cast<uint32_t>(a.splits - 1)) return;
    __threadfence();
    for (int i = tid; i < MB * kRowBlock; i += kLayerThreads) {
      const int b = i / kRowBlock;
      const int r = i - b * kRowBlock;
      float s = 0.f;
      for (int sp = 0; sp < a.splits; ++sp)
        s += __ldcg(a.partials + (static_cast<size_t>(sp) * MB + b) * a.m + rb * kRowBlock + r);
      zs[i] = s;
    }
    if (tid == 0) a.counters[rb] = 0u;  // leave the workspace zeroed for the next call
    __syncthreads();
  }

  // ---- epilogue: scale, output signs + FWHT, binary16 ----------------------
  for (int b = warp; b < MB; b += kLayerThreads / 32) {
    const int r0 = rb * kRowBlock + 4 * lane;
    float v[4], sc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = zs[b * kRowBlock + 4 * lane + j];
    load_half4(a.scales + r0, sc);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] *= sc[j];
    if (a.s_out != nullptr) {
      float s[4];
      load_half4(a.s_out + r0, s);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] *= s[j];
      fwht128_warp(v, lane);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
    }
    store_half4(a.y + static_cast<size_t>(b) * a.m + r0, v);
  }
}

template <int K, int CB, int MB>
exl3_status launch_layer_t(const LayerArgs& a, cudaStream_t stream) {
  const int nblk = a.n / kRowBlock;
  const int ns_max = ((nblk + a.splits - 1) / a.splits) * kRowBlock;
  const size_t smem = static_cast<size_t>(MB) * (ns_max + kRowBlock) * sizeof(float);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(layer_kernel<K, CB, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return EXL3_ERR_CUDA;
  }
  const dim3 grid(a.m / kRowBlock, a.splits);
  layer_kernel<K, CB, MB><<<grid, kLayerThreads, smem, stream>>>(a);
  return launch_status();
}

template <int K>
exl3_status launch_layer_dispatch(const LayerArgs& a, int mb, cudaStream_t stream) {
  if (a.codebook == kCb3Inst) {
    switch (mb) {
      case 1: return launch_layer_t<K, kCb3Inst, 1>(a, stream);
      case 2: return launch_layer_t<K, kCb3Inst, 2>(a, stream);
      case 4: return launch_layer_t<K, kCb3Inst, 4>(a, stream);
      case 8: return launch_layer_t<K, kCb3Inst, 8>(a, stream);
      default: return EXL3_ERR_BATCH;
    }
  }
  switch (mb) {
    case 1: return launch_layer_t<K, kCb1Mad, 1>(a, stream);
    case 2: return launch_layer_t<K, kCb1Mad, 2>(a, stream);
    case 4: return launch_layer_t<K, kCb1Mad, 4>(a, stream);
    case 8: return launch_layer_t<K, kCb1Mad, 8>(a, stream);
    default: return EXL3_ERR_BATCH;
  }
}

}  // namespace exl3

#define EXL3_DEFINE_LAYER_LAUNCHER(KK)                                                         \
  namespace exl3 {                                                                             \
  exl3_status launch_layer_k##KK(const LayerArgs& a, int mb, cudaStream_t stream) {            \
    return launch_layer_dispatch<KK>(a, mb, stream);                                           \
  }                                                                                            \
  }
