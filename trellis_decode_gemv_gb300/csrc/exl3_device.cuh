// Device-side building blocks shared by every libexl3 kernel: trellis window
// extraction, the two computed codes, and the 128-point Walsh-Hadamard
// butterfly.  Everything here is the GPU's own statement of the format; nothing
// is shared with the CPU oracle.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace exl3 {

// ---------------------------------------------------------------------------
// Codebook parameters (computed codes of "Trellis Quantization", Part nine).
// The pages print no constants for QTIP's generator; the LCG pair is the one
// printed in the conceptual decoder of "ExLlamaV3 & EXL3 Deep Dive" Section 3,
// the 3INST mask keeps sign + two low exponent bits + mantissa of each half and
// the magic pins the biased exponent to 12..15 (|half| in [1/8, 2)).
// ---------------------------------------------------------------------------
constexpr uint32_t kLcgMul = 0x9E3779B9u;
constexpr uint32_t kLcgAdd = 0x7F4A7C15u;
constexpr uint32_t k3InstMask = 0x8FFF8FFFu;
constexpr uint32_t k3InstMagic = 0x30003000u;
// 1MAD: four uniform bytes have mean 510 and variance 21845; the weight is
// (S - 510) times 1/sqrt(21845) rounded to binary32 (= 0x3BDDB446).
constexpr int kOneMadCentre = 510;
constexpr float kOneMadScale = 0x1.bb688cp-8f;
// 1/sqrt(128) rounded to binary32 (= 0x3DB504F3).
constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;

constexpr int kCb3Inst = 0;
constexpr int kCb1Mad = 1;

__device__ __forceinline__ uint32_t lcg(uint32_t s) { return s * kLcgMul + kLcgAdd; }

// (x & k3InstMask) ^ k3InstMagic as one three-input logic instruction
// (truth table 0x6A = (a & b) ^ c for a = 0xF0, b = 0xCC, c = 0xAA).
__device__ __forceinline__ uint32_t mask_xor_3inst(uint32_t x) {
  uint32_t h;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(h) : "r"(x), "r"(k3InstMask), "r"(k3InstMagic));
  return h;
}

// 3INST: LCG, mask+XOR into two binary16 halves (one LOP3), one binary16 add
// rounded to nearest even.
__device__ __forceinline__ __half code_3inst(uint32_t s) {
  const uint32_t h = mask_xor_3inst(lcg(s));
  const __half lo = __ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu));
  const __half hi = __ushort_as_half(static_cast<unsigned short>(h >> 16));
  return __hadd(lo, hi);
}

// 1MAD: LCG, byte sum S (one dp4a against 0x01010101), (S - 510) exact in
// binary32, one binary32 multiply, one rounding to binary16.
__device__ __forceinline__ __half code_1mad(uint32_t s) {
  const uint32_t x = lcg(s);
  const int S = static_cast<int>(__dp4a(x, 0x01010101u, 0u));
  const float c = static_cast<float>(S - kOneMadCentre);
  return __float2half_rn(__fmul_rn(c, kOneMadScale));
}

template <int CB>
__device__ __forceinline__ __half decode_state(uint32_t s) {
  if constexpr (CB == kCb3Inst) {
    return code_3inst(s);
  } else {
    return code_1mad(s);
  }
}

// ---------------------------------------------------------------------------
// Trellis windows ("Trellis Quantization", Part eight).
//
// A thread that owns rows 2p and 2p+1 of a tile owns steps 32p .. 32p+31, whose
// windows start at bits 32pK .. 32pK + 31K: word-aligned for every K, covering
// kPairWords words starting at word pK (circularly: the last pair wraps to the
// start of the tile's stream, which is the tail-biting sequence).
// ---------------------------------------------------------------------------
template <int K>
struct RowPair {
  static constexpr int kTileWords = 8 * K;
  static constexpr int kPairWords = (31 * K + 16 + 31) / 32;
};

template <int K>
__device__ __forceinline__ void load_row_pair(const uint32_t* __restrict__ tile, int p,
                                              uint32_t (&w)[RowPair<K>::kPairWords]) {
#pragma unroll
  for (int i = 0; i < RowPair<K>::kPairWords; ++i) {
    int idx = p * K + i;
    if (idx >= RowPair<K>::kTileWords) idx -= RowPair<K>::kTileWords;
    w[i] = __ldg(tile + idx);
  }
}

// State of step c (0..31, a compile-time constant after unrolling) of a row
// pair: the 16 bits starting at bit K*c of the words w (MSB first).
template <int K>
__device__ __forceinline__ uint32_t pair_state(const uint32_t (&w)[RowPair<K>::kPairWords], int c) {
  const int b = K * c;
  const int q = b >> 5;
  const int sh = b & 31;
  uint32_t v;
  if (sh == 0) {
    v = w[q];
  } else if (sh <= 16) {
    v = w[q] << sh;  // the window lies in word q
  } else {
    v = __funnelshift_l(w[q + 1], w[q], sh);
  }
  return v >> 16;
}

// The 32 bits of the stream starting at bit b (b compile-time), b + 31 within w.
template <int K>
__device__ __forceinline__ uint32_t pair_bits32(const uint32_t (&w)[RowPair<K>::kPairWords], int b) {
  const int q = b >> 5;
  const int sh = b & 31;
  return sh == 0 ? w[q] : __funnelshift_l(w[q + 1], w[q], sh);
}

// All 32 states of a row pair.  When K divides 16, the 32 bits starting at bit
// K*c hold both the window of step c (top half) and that of step c + 16/K
// (bottom half), so one funnel shift serves two states.
template <int K>
__device__ __forceinline__ void pair_states(const uint32_t (&w)[RowPair<K>::kPairWords],
                                            uint32_t (&s)[32]) {
  if constexpr (16 % K == 0) {
    constexpr int D = 16 / K;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if ((c / D) % 2 == 0) {
        const uint32_t r = pair_bits32<K>(w, K * c);
        s[c] = r >> 16;
        s[c + D] = r & 0xFFFFu;
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < 32; ++c) s[c] = pair_state<K>(w, c);
  }
}

// Weight of a state in fp32, for the fused product.
//  3INST: the binary16 sum of the two halves (exactly the defined weight),
//         widened to fp32.
//  1MAD:  the exact integer S - 510 as fp32, obtained without an int-to-float
//         conversion: dp4a adds the byte sum to the bit pattern of 1.5 * 2^23
//         minus 510, whose low mantissa bits then hold 1.5*2^23 + S - 510
//         exactly, and one subtraction removes the offset.  The 1/sqrt(21845)
//         factor is applied to x-tilde instead, so this skips the per-weight
//         binary16 rounding of the defined weight (a relative change of at most
//         2^-11 per weight, inside the layer tolerance).
constexpr uint32_t kOneMadMagicBits = 0x4B400000u - static_cast<uint32_t>(kOneMadCentre);
constexpr float kOneMadMagic = 12582912.0f;  // 1.5 * 2^23

template <int CB>
__device__ __forceinline__ float decode_f32(uint32_t s) {
  if constexpr (CB == kCb3Inst) {
    return __half2float(code_3inst(s));
  } else {
    const uint32_t x = lcg(s);
    return __uint_as_float(__dp4a(x, 0x01010101u, kOneMadMagicBits)) - kOneMadMagic;
  }
}

// Factor applied to x-tilde by the fused product for code CB (see decode_f32).
template <int CB>
__device__ __forceinline__ float x_factor() {
  return CB == kCb1Mad ? kOneMadScale : 1.0f;
}

// ---------------------------------------------------------------------------
// 128-point fast Walsh-Hadamard transform across one warp, 4 elements per lane
// (element e = 4*lane + j), unnormalized, Sylvester (natural) order:
// out_i = sum_j (-1)^popcount(i & j) in_j.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fwht128_warp(float (&v)[4], int lane) {
  {
    const float a0 = v[0] + v[1], a1 = v[0] - v[1];
    const float a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[2] = a0 - a2;
    v[1] = a1 + a3;
    v[3] = a1 - a3;
  }
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const bool upper = (lane & d) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float o = __shfl_xor_sync(0xFFFFFFFFu, v[j], d);
      v[j] = upper ? (o - v[j]) : (v[j] + o);
    }
  }
}

}  // namespace exl3
