// Device-side building blocks shared by every libexl3 kernel: trellis window
// extraction, the computed codes, and the 128-point Walsh-Hadamard
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

// (S - centre) exactly in binary32 for the byte sum S of x, without an
// int-to-float conversion: the dp4a adds S onto the bit pattern of 2^23
// (0x4B000000), which is then the binary32 value 2^23 + S exactly (S < 2^23),
// and subtracting 2^23 + centre is exact (the magic-number splice of
// "Trellis Quantization" Part three, in binary32).
__device__ __forceinline__ float centred_byte_sum(uint32_t x, int centre) {
  const float biased = __uint_as_float(__dp4a(x, 0x01010101u, 0x4B000000u));
  return __fsub_rn(biased, 8388608.0f + static_cast<float>(centre));
}

// 1MAD: LCG, byte sum S (one dp4a against 0x01010101), (S - 510) exact in
// binary32, one binary32 multiply, one rounding to binary16.
__device__ __forceinline__ __half code_1mad(uint32_t s) {
  return __float2half_rn(__fmul_rn(centred_byte_sum(lcg(s), kOneMadCentre), kOneMadScale));
}

// MCG and mul1, EXL3's later codes ("Trellis Quantization", Parts eleven and
// twelve): the generator keeps only the multiply (the pages do not print the
// multiplier they adopt; the LCG multiplier above is used).  MCG is 3INST on
// that generator; mul1 masks every byte of the product to six bits, sums the
// four bytes (mean 4 * 31.5 = 126, variance 4 * (64^2 - 1) / 12 = 1365),
// subtracts 126 and scales by 1/sqrt(1365) rounded to binary32 (= 0x3CDDBAC5).
constexpr int kCbMcg = 2;
constexpr int kCbMul1 = 3;
constexpr uint32_t kMul1Mask = 0x3F3F3F3Fu;
constexpr int kMul1Centre = 126;
constexpr float kMul1Scale = 0x1.bb758ap-6f;

__device__ __forceinline__ uint32_t mcg(uint32_t s) { return s * kLcgMul; }

// Generator output of code CB for state s.
template <int CB>
__device__ __forceinline__ uint32_t generate(uint32_t s) {
  if constexpr (CB == kCbMcg || CB == kCbMul1) {
    return mcg(s);
  } else {
    return lcg(s);
  }
}

// Codes whose weight is an affine function of a byte sum (1MAD, mul1): the
// word whose bytes are summed, the centre and the scale.
template <int CB>
__host__ __device__ constexpr bool byte_sum_code() {
  return CB == kCb1Mad || CB == kCbMul1;
}
template <int CB>
__device__ __forceinline__ uint32_t summed_bytes(uint32_t x) {
  if constexpr (CB == kCbMul1) {
    return x & kMul1Mask;
  } else {
    return x;
  }
}
template <int CB>
__host__ __device__ constexpr int byte_sum_centre() {
  return CB == kCbMul1 ? kMul1Centre : kOneMadCentre;
}
template <int CB>
__host__ __device__ constexpr float byte_sum_scale() {
  return CB == kCbMul1 ? kMul1Scale : kOneMadScale;
}

// MCG: the three-instruction code on the multiplicative generator.
__device__ __forceinline__ __half code_mcg(uint32_t s) {
  const uint32_t h = mask_xor_3inst(mcg(s));
  const __half lo = __ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu));
  const __half hi = __ushort_as_half(static_cast<unsigned short>(h >> 16));
  return __hadd(lo, hi);
}

// mul1: masked byte sum S (one dp4a), (S - 126) exact in binary32, one binary32
// multiply, one rounding to binary16.
__device__ __forceinline__ __half code_mul1(uint32_t s) {
  return __float2half_rn(__fmul_rn(centred_byte_sum(mcg(s) & kMul1Mask, kMul1Centre), kMul1Scale));
}

// The defined binary16 weights of two states, packed (s0 in the low half):
// the same roundings as decode_state, two at a time (one paired conversion,
// or one packed add for the three-instruction codes).
template <int CB>
__device__ __forceinline__ uint32_t decode_pair(uint32_t s0, uint32_t s1);

template <int CB>
__device__ __forceinline__ __half decode_state(uint32_t s) {
  if constexpr (CB == kCb3Inst) {
    return code_3inst(s);
  } else if constexpr (CB == kCb1Mad) {
    return code_1mad(s);
  } else if constexpr (CB == kCbMcg) {
    return code_mcg(s);
  } else {
    return code_mul1(s);
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

// Factor applied to x-tilde by the fused products: the byte-sum codes
// multiply x by the exact integer (S - centre) and take their scale from x,
// which skips the per-weight binary16 rounding of the defined weight (a
// relative change of at most 2^-11 per weight, inside the layer tolerance).
template <int CB>
__host__ __device__ constexpr float x_factor() {
  if constexpr (byte_sum_code<CB>()) {
    return byte_sum_scale<CB>();
  } else {
    return 1.0f;
  }
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

template <int CB>
__device__ __forceinline__ uint32_t decode_pair(uint32_t s0, uint32_t s1) {
  if constexpr (CB == kCb1Mad || CB == kCbMul1) {
    constexpr int centre = CB == kCbMul1 ? kMul1Centre : kOneMadCentre;
    constexpr float scale = CB == kCbMul1 ? kMul1Scale : kOneMadScale;
    const uint32_t x0 = CB == kCbMul1 ? (mcg(s0) & kMul1Mask) : lcg(s0);
    const uint32_t x1 = CB == kCbMul1 ? (mcg(s1) & kMul1Mask) : lcg(s1);
    const __half2 w = __floats2half2_rn(__fmul_rn(centred_byte_sum(x0, centre), scale),
                                        __fmul_rn(centred_byte_sum(x1, centre), scale));
    return *reinterpret_cast<const uint32_t*>(&w);
  } else {
    const uint32_t h0 = mask_xor_3inst(CB == kCbMcg ? mcg(s0) : lcg(s0));
    const uint32_t h1 = mask_xor_3inst(CB == kCbMcg ? mcg(s1) : lcg(s1));
    const uint32_t lo = __byte_perm(h0, h1, 0x5410);  // (lo0, lo1)
    const uint32_t hi = __byte_perm(h0, h1, 0x7632);  // (hi0, hi1)
    const __half2 w = __hadd2(*reinterpret_cast<const __half2*>(&lo), *reinterpret_cast<const __half2*>(&hi));
    return *reinterpret_cast<const uint32_t*>(&w);
  }
}

}  // namespace exl3
