// The int8-activation layer kernel ("Trellis Quantization" Part eleven: with
// the activations quantized to eight-bit integers and the weight an affine
// function of a byte sum, one dp4a computes code value times activation for
// the four bytes at once, so decode and multiply fuse into one integer
// instruction).
//
// For the byte-sum codes (1MAD, mul1) the weight is C * (S - centre), S the
// sum of the four (masked) bytes of the generator output.  With q_j the int8
// activation replicated into the four bytes of a word, dp4a(bytes, q_j, acc)
// adds S * q_j exactly, so over a 16-column tile a row accumulates
// sum_j S_j q_j in int32 and
//     z += (C * qscale_block) * (acc - centre * sum_j q_j)
// once per tile.  Per weight: the window, one multiply(-add) for the
// generator, (mul1: one AND for the six-bit mask), one dp4a.
//
// Same lane mapping and work split as the warp-shuffle sub-unit kernel: a
// warp decodes one tile row, lane 8 * jt + p takes rows 2p, 2p + 1 of tiles
// jt, jt + 4, ... of a sub-unit of 4 * TPL consecutive tiles (unrolled); one
// CTA per SM, sub-units interleaved over the warps of all CTAs (the sub-units
// of the layers of a group are numbered one after the other); shuffles combine
// the four tile groups and fp32 reductions add each row's sum into the
// workspace row sums.
#pragma once

#include "exl3_device.cuh"
#include "exl3_host.cuh"
#include "exl3_layer.cuh"

namespace exl3 {

// dp4a of four unsigned bytes with four signed bytes (1MAD's full bytes).
__device__ __forceinline__ int dp4a_u8s8(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <int CB>
__device__ __forceinline__ int byte_dot(uint32_t x, int q4, int acc) {
  if constexpr (CB == kCbMul1) {
    return __dp4a(static_cast<int>(x & kMul1Mask), q4, acc);  // bytes <= 63: signed dp4a
  } else {
    return dp4a_u8s8(x, q4, acc);
  }
}

// Sub-unit lu of layer a (lane 8*jt + p): tiles J0 + jt + 4t (t < TPL), rows
// 2p, 2p+1 of each; code words two tiles ahead, addressed from one per-lane
// pointer (and one for the last row pair's wrapped words), as in the binary16
// sub-unit kernel.
template <int K, int CB, int MB, int TPL>
__device__ __forceinline__ void i8_unit(const I8Layer& a, int lu, int lane, bool& waited) {
  const int jt = lane >> 3;
  const int p = lane & 7;
  constexpr int kTw = RowPair<K>::kTileWords;
  constexpr int kPw = RowPair<K>::kPairWords;
  const int nt = a.n / 16;
  const int I = a.row_magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(lu), a.row_magic)) : lu / a.per_row;
  const int J0 = (lu - I * a.per_row) * (4 * TPL) + jt;  // this lane's first tile
  const uint32_t* tp = a.codes + (static_cast<size_t>(I) * nt + J0) * kTw;
  const uint32_t* lp = tp + p * K;
  const uint32_t* lw = lp - (p == 7 ? kTw : 0);
  auto load_pair = [&](int toff, uint32_t (&wd)[kPw]) {
#pragma unroll
    for (int i = 0; i < kPw; ++i) wd[i] = __ldg((i < K ? lp : lw) + toff + i);
  };
  uint32_t w[2][kPw];
  if (J0 < nt) load_pair(0, w[0]);
  if (TPL > 1 && J0 + 4 < nt) load_pair(4 * kTw, w[1]);
  // The activation words, tile corrections and block factors come from the
  // preceding grid on the stream; the code words above do not.
  if (!waited) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    waited = true;
  }

  float acc[MB][2];
#pragma unroll
  for (int b = 0; b < MB; ++b) acc[b][0] = acc[b][1] = 0.f;

#pragma unroll
  for (int t = 0; t < TPL; ++t) {
    const int J = J0 + 4 * t;
    if (J < nt) {  // all lanes but on a row's ragged last sub-unit
      uint32_t gen[32];
      pair_generate<K, CB>(w[t & 1], gen);
      if (t + 2 < TPL && J + 8 < nt) load_pair((4 * t + 8) * kTw, w[t & 1]);
      const int4* qrow = reinterpret_cast<const int4*>(a.q4 + static_cast<size_t>(J) * 16);
      int ia[MB], ib[MB];
#pragma unroll
      for (int b = 0; b < MB; ++b) ia[b] = ib[b] = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int4 qv[MB];
#pragma unroll
        for (int b = 0; b < MB; ++b) qv[b] = qrow[static_cast<size_t>(b) * (a.n / 4) + q];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * q + j;
#pragma unroll
          for (int b = 0; b < MB; ++b) {
            const int qw = j == 0 ? qv[b].x : j == 1 ? qv[b].y : j == 2 ? qv[b].z : qv[b].w;
            ia[b] = byte_dot<CB>(gen[c], qw, ia[b]);
            ib[b] = byte_dot<CB>(gen[16 + c], qw, ib[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < MB; ++b) {
        const int corr = a.tcorr[static_cast<size_t>(b) * nt + J];
        const float f = a.cs[static_cast<size_t>(b) * (a.n / kRowBlock) + J / 8];
        acc[b][0] = fmaf(f, static_cast<float>(ia[b] - corr), acc[b][0]);
        acc[b][1] = fmaf(f, static_cast<float>(ib[b] - corr), acc[b][1]);
      }
    }
  }

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
      float* z = a.zacc + static_cast<size_t>(b) * a.m + I * 16 + 2 * p;
      atomicAdd(z, acc[b][0]);
      atomicAdd(z + 1, acc[b][1]);
    }
  }
}

// Warps per CTA: 32 at batch 1; batch 2 keeps 16 (its byte-dot sums and
// activation words do not fit 64 registers at four tiles a lane).
template <int MB>
constexpr int i8_warps() { return MB == 1 ? 32 : MB <= 4 ? 16 : 8; }

// Warp w of CTA b takes the sub-units w * grid + b + i * (grid * warps).
template <int K, int CB, int MB, int TPL>
__global__ void __launch_bounds__(32 * i8_warps<MB>(), 1) i8_kernel(const I8Args g) {
  constexpr int kWarps = i8_warps<MB>();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const long long stride = static_cast<long long>(gridDim.x) * kWarps;
  // The output kernel may be scheduled now (it waits for this grid to finish).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  bool waited = false;
  // CTA-fastest numbering: the last partial round falls on every SM alike
  long long u = static_cast<long long>(warp) * gridDim.x + blockIdx.x;
  if (u >= g.units) return;
  int li = 0;
  {
    int hi = g.count - 1;  // the last layer whose first sub-unit is <= u
    while (li < hi) {
      const int mid = (li + hi + 1) >> 1;
      if (u >= g.l[mid].u_begin) li = mid; else hi = mid - 1;
    }
  }
  for (; u < g.units; u += stride) {
    // a warp's sub-units increase, so its layer index only moves forward
    while (li + 1 < g.count && u >= g.l[li + 1].u_begin) ++li;
    const I8Layer& a = g.l[li];
    i8_unit<K, CB, MB, TPL>(a, static_cast<int>(u - a.u_begin), lane, waited);
  }
}

// The sub-units of code CB (up to `end`) of a one-K kernel, continuing the
// warp's sequence u; returns where it stopped.
template <int K, int CB>
__device__ __forceinline__ long long i8_kset_loop(const I8Args& g, long long u, long long stride, long long end,
                                                  int& li, int lane, bool& waited) {
  for (; u < end; u += stride) {
    while (li + 1 < g.count && u >= g.l[li + 1].u_begin) ++li;
    const I8Layer& a = g.l[li];
    i8_unit<K, CB, 1, 8>(a, static_cast<int>(u - a.u_begin), lane, waited);
  }
  return u;
}

// Batch 1, 32-tile sub-units: the 1MAD and mul1 layers of one K, ordered by
// code, in one launch, as the binary16 one-K kernel.
template <int K>
__global__ void __launch_bounds__(32 * i8_warps<1>(), 1) i8_kernel_kset(const I8Args g) {
  constexpr int kWarps = i8_warps<1>();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const long long stride = static_cast<long long>(gridDim.x) * kWarps;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  bool waited = false;
  long long u = static_cast<long long>(warp) * gridDim.x + blockIdx.x;
  if (u >= g.units) return;
  int li = 0;
  {
    int hi = g.count - 1;  // the last layer whose first sub-unit is <= u
    while (li < hi) {
      const int mid = (li + hi + 1) >> 1;
      if (u >= g.l[mid].u_begin) li = mid; else hi = mid - 1;
    }
  }
  u = i8_kset_loop<K, kCb1Mad>(g, u, stride, g.class_end[0], li, lane, waited);
  i8_kset_loop<K, kCbMul1>(g, u, stride, g.class_end[1], li, lane, waited);
}

template <int K>
exl3_status launch_i8_kset_t(const I8Args& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.ctas));
  cfg.blockDim = dim3(32 * i8_warps<1>());
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, i8_kernel_kset<K>, a) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

template <int K, int CB, int MB, int TPL>
exl3_status launch_i8_t(const I8Args& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.ctas));
  cfg.blockDim = dim3(32 * i8_warps<MB>());
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, i8_kernel<K, CB, MB, TPL>, a) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

template <int K, int CB, int MB>
exl3_status launch_i8_mb(const I8Args& a, cudaStream_t stream) {
  switch (a.sub) {
    case 32:
      if constexpr (MB == 1) return launch_i8_t<K, CB, MB, 8>(a, stream);
      return EXL3_ERR_BATCH;
    case 16: return launch_i8_t<K, CB, MB, 4>(a, stream);
    case 8: return launch_i8_t<K, CB, MB, 2>(a, stream);
    default: return launch_i8_t<K, CB, MB, 1>(a, stream);
  }
}

template <int K, int CB>
exl3_status launch_i8_cb(const I8Args& a, int mb, cudaStream_t stream) {
  switch (mb) {
    case 1: return launch_i8_mb<K, CB, 1>(a, stream);
    case 2: return launch_i8_mb<K, CB, 2>(a, stream);
    case 4: return launch_i8_mb<K, CB, 4>(a, stream);
    case 8: return launch_i8_mb<K, CB, 8>(a, stream);
    default: return EXL3_ERR_BATCH;
  }
}

template <int K>
exl3_status launch_i8_dispatch(const I8Args& a, int codebook, int mb, cudaStream_t stream) {
  switch (codebook) {
    case kCb1Mad: return launch_i8_cb<K, kCb1Mad>(a, mb, stream);
    case kCbMul1: return launch_i8_cb<K, kCbMul1>(a, mb, stream);
    default: return EXL3_ERR_CODEBOOK;
  }
}

}  // namespace exl3

#define EXL3_DEFINE_I8_LAUNCHER(KK)                                                     \
  namespace exl3 {                                                                      \
  exl3_status launch_i8_k##KK(const I8Args& a, int codebook, int mb, cudaStream_t stream) { \
    return launch_i8_dispatch<KK>(a, codebook, mb, stream);                             \
  }                                                                                     \
  exl3_status launch_i8_kset_k##KK(const I8Args& a, cudaStream_t stream) {              \
    return launch_i8_kset_t<KK>(a, stream);                                             \
  }                                                                                     \
  }
