// Fused layer kernel, warp-shuffle path (batch 1..8):
//   y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x))))
// ("ExLlamaV3 & EXL3 Deep Dive" Section 2 runtime identity; W-hat decoded on
// the fly from the bitshift-trellis codes of "Trellis Quantization" Parts
// eight and nine; blockwise 128-point transforms of Part eleven).
//
// Each call runs two kernels on the stream, chained by programmatic dependent
// launch (the second starts while the first runs and waits for it,
// griddepcontrol.wait, before reading what it writes):
//  1. layer_kernel (below) accumulates W-hat x-tilde into the fp32 row sums
//     zacc with atomic adds;
//  2. epi_kernel (csrc/exl3_rht_decode.cu) applies the scale, the output signs
//     and the 128-point FWHT to each 128-row block of zacc, stores y as
//     binary16 and zeroes zacc for the next call.
//
// Work split (stream-K style): the (m/128 row blocks) x (n/16 tile columns)
// work units are cut into gridDim.x equal contiguous ranges, one per CTA; a
// range is a sequence of segments, each inside one row block.  8 warps per
// CTA, warp w owns tile-row 8*rb + w of the segment's row block; lane
// 8*jt + p handles every 4th tile (jt) and the row pair 2p, 2p+1 of the tile,
// so each thread decodes 32 consecutive trellis steps from a word-aligned
// window (code words are loaded two tiles ahead of their decode).  Each
// segment starts by rotating the x columns it needs into shared memory (signs,
// 128-point FWHT across a warp, 1/sqrt(128), times the code's x factor,
// rounded to binary16, duplicated into both halves of a 32-bit word), one
// warp per overlapping 128-block.  Per column one packed binary16
// FMA (HFMA2):
//   3INST  acc += (lo, hi) * (x, x)   -- the two halves of the mask/XOR step,
//          so lo*x + hi*x is the weight times x without a separate add;
//   1MAD   acc += (S_a - 510, S_b - 510) * (x, x) for rows 2p and 2p+1, the
//          byte sums spliced into binary16 1024 + S by dp4a, paired with one
//          byte permute and made exact with one packed subtraction of 1534.
// The packed accumulators are flushed into fp32 after every 16 columns (one
// tile row), which keeps the binary16 accumulation error near 1e-3 of a
// tile-row partial sum and about 7e-4 of the result (relative L2).
//
// Combine: a warp-shuffle reduction over the 4 tile groups and fp32 atomic adds
// of each segment's row sums into zacc.  No CTA waits on another; the kernel
// boundary orders the sums before the epilogue kernel.  The atomic adds make
// the fp32 summation order, and so the last bit of some outputs, vary from
// run to run.
#pragma once

#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {

constexpr int kLayerThreads = 256;
// Longest segment (tile columns) handled between two shared-memory refills of
// the rotated x.
constexpr int kSegTiles = 64;

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

// Resident 256-thread CTAs per SM the kernel is compiled for (registers).
template <int MB>
__host__ __device__ constexpr int layer_ctas_per_sm() {
  return MB == 1 ? 5 : MB == 2 ? 4 : 1;
}

template <int K, int CB, int MB>
__global__ void __launch_bounds__(kLayerThreads, layer_ctas_per_sm<MB>()) layer_kernel(LayerArgs a) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int jt = lane >> 3;
  const int p = lane & 7;
  constexpr int kTw = RowPair<K>::kTileWords;
  const int nt = a.n / 16;
  const long long units = static_cast<long long>(a.m / kRowBlock) * nt;
  const long long u_begin = static_cast<long long>(blockIdx.x) * units / gridDim.x;
  const long long u_end = static_cast<long long>(blockIdx.x + 1) * units / gridDim.x;
  const __half2 k1534 = __half2half2(__ushort_as_half(0x65FE));  // 1534 = 1024 + 510
  __shared__ uint4 xs[MB * kSegTiles * 4];  // rotated x of the segment, [MB][tiles][4]

  // The output kernel may be scheduled now (it waits for this grid to finish).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  bool waited = false;
  for (long long u = u_begin; u < u_end;) {
    const int rb = static_cast<int>(u / nt);
    const int ja = static_cast<int>(u - static_cast<long long>(rb) * nt);
    const long long left = u_end - u;
    const int span = left < kSegTiles ? static_cast<int>(left) : kSegTiles;
    const int jb = ja + span < nt ? ja + span : nt;
    const int I = rb * (kRowBlock / 16) + warp;
    const uint32_t* rowp = a.codes + static_cast<size_t>(I) * nt * kTw;

    // Code words are loaded two tiles ahead of their decode; the first two are
    // requested before the segment's x rotation.
    int J = ja + jt;
    uint32_t w0[RowPair<K>::kPairWords], w1[RowPair<K>::kPairWords];
    if (J < jb) load_row_pair<K>(rowp + static_cast<size_t>(J) * kTw, p, w0);
    if (J + 4 < jb) load_row_pair<K>(rowp + static_cast<size_t>(J + 4) * kTw, p, w1);
    // x (and the zeroed row sums) come from the preceding grids on the stream;
    // the codes above do not.
    if (!waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }

    // Rotate the x columns of the segment into shared memory: every 128-block
    // that overlaps it, one warp per (batch row, block): signs, 128-point FWHT,
    // 1/sqrt(128), the code's x factor, binary16, duplicated in both halves.
    __syncthreads();  // the previous segment's readers are done
    {
      const int c_lo = ja * 16;
      const int c_hi = jb * 16;
      const int kb0 = c_lo / kRowBlock;
      const int nkb = (c_hi - 1) / kRowBlock - kb0 + 1;
      for (int job = warp; job < MB * nkb; job += kLayerThreads / 32) {
        const int b = job / nkb;
        const int col = (kb0 + job - b * nkb) * kRowBlock + 4 * lane;
        float v[4];
        load_half4(a.x + static_cast<size_t>(b) * a.n + col, v);
        if (a.s_in != nullptr) {
          float sg[4];
          load_half4(a.s_in + col, sg);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] *= sg[j];
          fwht128_warp(v, lane);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
        }
        if (col >= c_lo && col < c_hi) {
          uint4 pk;
          pk.x = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[0] * x_factor<CB>()))) * 0x10001u;
          pk.y = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[1] * x_factor<CB>()))) * 0x10001u;
          pk.z = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[2] * x_factor<CB>()))) * 0x10001u;
          pk.w = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[3] * x_factor<CB>()))) * 0x10001u;
          xs[b * kSegTiles * 4 + (col - c_lo) / 4] = pk;
        }
      }
    }
    __syncthreads();

    float acc[MB][2];
#pragma unroll
    for (int b = 0; b < MB; ++b) acc[b][0] = acc[b][1] = 0.f;

    while (J < jb) {
      uint32_t st[32];
      pair_states<K>(w0, st);
#pragma unroll
      for (int i = 0; i < RowPair<K>::kPairWords; ++i) w0[i] = w1[i];
      if (J + 8 < jb) load_row_pair<K>(rowp + static_cast<size_t>(J + 8) * kTw, p, w1);
      const uint4* xrow = xs + (J - ja) * 4;
      J += 4;
      __half2 ha[MB], hb[MB];
#pragma unroll
      for (int b = 0; b < MB; ++b) {
        ha[b] = __float2half2_rn(0.f);
        hb[b] = __float2half2_rn(0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 xv[MB];
#pragma unroll
        for (int b = 0; b < MB; ++b) xv[b] = xrow[b * kSegTiles * 4 + q];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * q + j;
          const uint32_t xa = lcg(st[c]);
          const uint32_t xb = lcg(st[16 + c]);
          if constexpr (CB == kCb3Inst) {
            const uint32_t pa = mask_xor_3inst(xa);
            const uint32_t pb = mask_xor_3inst(xb);
#pragma unroll
            for (int b = 0; b < MB; ++b) {
              const uint32_t xw = j == 0 ? xv[b].x : j == 1 ? xv[b].y : j == 2 ? xv[b].z : xv[b].w;
              const __half2 x2 = *reinterpret_cast<const __half2*>(&xw);
              ha[b] = __hfma2(*reinterpret_cast<const __half2*>(&pa), x2, ha[b]);
              hb[b] = __hfma2(*reinterpret_cast<const __half2*>(&pb), x2, hb[b]);
            }
          } else {
            const uint32_t ra = __dp4a(xa, 0x01010101u, 0x6400u);
            const uint32_t rb2 = __dp4a(xb, 0x01010101u, 0x6400u);
            const uint32_t pr = __byte_perm(ra, rb2, 0x5410);  // (1024 + S_a, 1024 + S_b)
            const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&pr), k1534);
#pragma unroll
            for (int b = 0; b < MB; ++b) {
              const uint32_t xw = j == 0 ? xv[b].x : j == 1 ? xv[b].y : j == 2 ? xv[b].z : xv[b].w;
              ha[b] = __hfma2(v, *reinterpret_cast<const __half2*>(&xw), ha[b]);
            }
          }
        }
      }
#pragma unroll
      for (int b = 0; b < MB; ++b) {
        if constexpr (CB == kCb3Inst) {
          acc[b][0] += __low2float(ha[b]) + __high2float(ha[b]);
          acc[b][1] += __low2float(hb[b]) + __high2float(hb[b]);
        } else {
          acc[b][0] += __low2float(ha[b]);
          acc[b][1] += __high2float(ha[b]);
        }
      }
    }

    // ---- warp-shuffle reduction over the 4 tile groups, accumulate into zacc --
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
        float* z = a.zacc + static_cast<size_t>(b) * a.m + rb * kRowBlock + warp * 16 + 2 * p;
        atomicAdd(z, acc[b][0]);
        atomicAdd(z + 1, acc[b][1]);
      }
    }
    u += jb - ja;
  }
}

template <int K, int CB, int MB>
exl3_status launch_layer_t(const LayerArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.ctas));
  cfg.blockDim = dim3(kLayerThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, layer_kernel<K, CB, MB>, a) != cudaSuccess) return EXL3_ERR_CUDA;
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
