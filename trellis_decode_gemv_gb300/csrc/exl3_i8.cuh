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
// jt, jt + 4, ... of a sub-unit of consecutive tiles; one CTA per SM, the warps
// take sub-units from a shared counter (the sub-units of up to four layers of
// a group are numbered one after the other); shuffles combine the four tile
// groups and fp32 reductions add each row's sum into the workspace row sums.
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

template <int K, int CB, int MB>
__device__ __forceinline__ void i8_body(const I8Args& g) {
  constexpr int kWarps = layer_warps<MB>();
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int jt = lane >> 3;
  const int p = lane & 7;
  constexpr int kTw = RowPair<K>::kTileWords;
  const int S = g.sub;
  const long long units = g.units;
  const int u_lo = static_cast<int>(units * blockIdx.x / gridDim.x);
  const int u_hi = static_cast<int>(units * (blockIdx.x + 1) / gridDim.x);
  __shared__ int next_unit;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) next_unit = 0;
  __syncthreads();

  bool waited = false;
  int u = u_lo + warp;
  while (u < u_hi) {
    // the layer of sub-unit u, then its tile row and first tile column
    int li = 0;
    {
      int hi = g.count - 1;  // the last layer whose first sub-unit is <= u
      while (li < hi) {
        const int mid = (li + hi + 1) >> 1;
        if (u >= g.l[mid].u_begin) li = mid; else hi = mid - 1;
      }
    }
    const I8Layer& a = g.l[li];
    const int nt = a.n / 16;
    const int lu = u - a.u_begin;
    const int I = lu / a.per_row;
    const int J0 = (lu - I * a.per_row) * S;
    const int J1 = J0 + S < nt ? J0 + S : nt;
    const uint32_t* rowp = a.codes + static_cast<size_t>(I) * nt * kTw;

    int J = J0 + jt;
    uint32_t w0[RowPair<K>::kPairWords], w1[RowPair<K>::kPairWords];
    if (J < J1) load_row_pair<K>(rowp + static_cast<size_t>(J) * kTw, p, w0);
    if (J + 4 < J1) load_row_pair<K>(rowp + static_cast<size_t>(J + 4) * kTw, p, w1);
    // The activation words, tile corrections and block factors come from the
    // preceding grid on the stream; the code words above do not.
    if (!waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }
    int un = 0;
    if (lane == 0) un = u_lo + kWarps + atomicAdd(&next_unit, 1);
    un = __shfl_sync(0xFFFFFFFFu, un, 0);

    float acc[MB][2];
#pragma unroll
    for (int b = 0; b < MB; ++b) acc[b][0] = acc[b][1] = 0.f;

    while (J < J1) {
      uint32_t st[32];
      pair_states<K>(w0, st);
#pragma unroll
      for (int i = 0; i < RowPair<K>::kPairWords; ++i) w0[i] = w1[i];
      if (J + 8 < J1) load_row_pair<K>(rowp + static_cast<size_t>(J + 8) * kTw, p, w1);
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
          const uint32_t xa = generate<CB>(st[c]);
          const uint32_t xb = generate<CB>(st[16 + c]);
#pragma unroll
          for (int b = 0; b < MB; ++b) {
            const int qw = j == 0 ? qv[b].x : j == 1 ? qv[b].y : j == 2 ? qv[b].z : qv[b].w;
            ia[b] = byte_dot<CB>(xa, qw, ia[b]);
            ib[b] = byte_dot<CB>(xb, qw, ib[b]);
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
      J += 4;
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
    u = un;
  }
}

template <int K, int CB, int MB>
__global__ void __launch_bounds__(32 * layer_warps<MB>(), 1) i8_kernel(const I8Args a) {
  i8_body<K, CB, MB>(a);
}

template <int K, int CB, int MB>
exl3_status launch_i8_t(const I8Args& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.ctas));
  cfg.blockDim = dim3(32 * layer_warps<MB>());
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, i8_kernel<K, CB, MB>, a) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

template <int K, int CB>
exl3_status launch_i8_cb(const I8Args& a, int mb, cudaStream_t stream) {
  switch (mb) {
    case 1: return launch_i8_t<K, CB, 1>(a, stream);
    case 2: return launch_i8_t<K, CB, 2>(a, stream);
    case 4: return launch_i8_t<K, CB, 4>(a, stream);
    case 8: return launch_i8_t<K, CB, 8>(a, stream);
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
  }
