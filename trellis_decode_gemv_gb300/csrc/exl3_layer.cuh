// Fused layer kernel, warp-shuffle path (batch 1..8):
//   y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x))))
// ("ExLlamaV3 & EXL3 Deep Dive" Section 2 runtime identity; W-hat decoded on
// the fly from the bitshift-trellis codes of "Trellis Quantization" Parts
// eight and nine; blockwise 128-point transforms of Part eleven).
//
// Two kernel designs share the decode and MAC below; the launch plan picks
// the sub-unit kernel for layers with at least about 1024 tiles per SM and the
// segment kernel (further down, which rotates x itself) for smaller ones.
// With the sub-unit kernel a call runs three kernels on the stream, chained by
// programmatic dependent launch (each starts while its predecessor runs and
// waits for it, griddepcontrol.wait, before reading what it writes):
//  1. xdup_kernel (csrc/exl3_rht_decode.cu) writes x-tilde = Hb(s_in (.) x),
//     times the code's x factor, as binary16 duplicated into both halves of a
//     32-bit word ("x pairs"), [mb][n];
//  2. layer_kernel (below) accumulates W-hat x-tilde into the fp32 row sums
//     zacc with atomic adds;
//  3. epi_kernel (csrc/exl3_rht_decode.cu) applies the scale, the output signs
//     and the 128-point FWHT to each 128-row block of zacc, stores y as
//     binary16 and zeroes zacc for the next call.
//
// Work split: a sub-unit is up to S (32, 16, 8 or 4; 32 at batch 1 only)
// consecutive tiles of one tile row; one CTA per SM; warp w of CTA b takes the
// sub-units w * grid + b + i * (grid * warps), each warp's tile row found by
// a multiply-high with a per-layer magic number and its layer by stepping
// forward from the one of its previous sub-unit.  In grouped calls the
// sub-units of every layer of the call are numbered one after the other; at
// batch 1 the layers of several codes of one K can share one launch
// (layer_kernel_kset, one loop per code).  In a sub-unit, lane 8*jt + p
// handles tiles J0 + jt, J0 + jt + 4, ... and the row pair 2p, 2p+1 of each:
// 32 consecutive
// trellis steps from a word-aligned window per tile (code words loaded two
// tiles ahead of their decode), with the x pairs of the tile's 16 columns read
// from L1/L2.  Per column one packed binary16 FMA (HFMA2):
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
// of each sub-unit's 16 row sums into zacc.  No CTA waits on another; the
// kernel boundary orders the sums before the epilogue kernel.  The atomic adds
// make the fp32 summation order, and so the last bit of some outputs, vary
// from run to run.
#pragma once

#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {

// ---- segment kernel (layers with under about 1024 tiles per SM) ------------
// Five 256-thread CTAs per SM at batch 1 (four at 2).  The (m/128 row blocks)
// x (n/16 tile columns) work units are cut into gridDim.x equal contiguous
// ranges, one per CTA; a range is a sequence of segments inside one row block.
// Warp w owns tile row w of the segment's row block, lane 8*jt + p tiles
// ja + jt, ja + jt + 4, ... and row pair 2p, 2p+1.  Each segment starts by
// rotating the x columns it needs into shared memory (one warp per overlapping
// 128-block: signs, FWHT, 1/sqrt(128), x factor, binary16 pairs), so no
// separate x-pair kernel runs; the decode and MAC are those of the sub-unit
// kernel below.
constexpr int kSegThreads = 256;
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
__host__ __device__ constexpr int seg_ctas_per_sm() {
  return MB == 1 ? 5 : MB == 2 ? 4 : 1;
}

template <int K, int CB, int MB>
__global__ void __launch_bounds__(kSegThreads, seg_ctas_per_sm<MB>()) seg_layer_kernel(LayerArgs a) {
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
  // binary16 of 1024 + the byte-sum centre (1534 for 1MAD, 1150 for mul1)
  const __half2 k1534 = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6400 + byte_sum_centre<CB>())));
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
      for (int job = warp; job < MB * nkb; job += kSegThreads / 32) {
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
          const uint32_t xa = generate<CB>(st[c]);
          const uint32_t xb = generate<CB>(st[16 + c]);
          if constexpr (!byte_sum_code<CB>()) {
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
            const uint32_t ra = __dp4a(summed_bytes<CB>(xa), 0x01010101u, 0x6400u);
            const uint32_t rb2 = __dp4a(summed_bytes<CB>(xb), 0x01010101u, 0x6400u);
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
        if constexpr (!byte_sum_code<CB>()) {
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

// ---- sub-unit kernel (larger layers) -------------------------------------------

// Warps of the one CTA per SM: 32 (1024 threads) at batch 1 and 2 (64
// registers: 24 warps with more registers measured 3-5% slower at batch 2),
// 16 for chunks of 4, 8 for 8 (registers).
template <int MB>
__host__ __device__ constexpr int layer_warps() {
  return MB <= 2 ? 32 : MB == 4 ? 16 : 8;
}
// Registers per thread of the batch-1 kernel.  For K <= 3, 56 x 1024 leaves
// 8192 of the SM's 65536 registers, room for one 128-thread CTA of the output
// kernel to be resident, waiting, when the layer kernel finishes (the batch-2
// kernel, 768 x 80, leaves 4096); wider code words need all 64.
template <int K>
__host__ __device__ constexpr int layer_max_regs() {
  return K <= 3 ? 56 : 64;
}

// Generator outputs of the 32 steps of a row pair (rows 2p, 2p+1 of a tile):
// the windows at bits K*c of the pair's words w.  When K divides 16 one
// 32-bit funnel word r holds the windows of steps c (top half) and c + 16/K
// (bottom half): one funnel shift, a shift and a mask for two windows.
template <int K, int CB>
__device__ __forceinline__ void pair_generate(const uint32_t (&w)[RowPair<K>::kPairWords], uint32_t (&g)[32]) {
  constexpr uint32_t kAdd = (CB == kCbMcg || CB == kCbMul1) ? 0u : kLcgAdd;
  if constexpr (16 % K == 0) {
    constexpr int D = 16 / K;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if ((c / D) % 2 == 0) {
        const uint32_t r = pair_bits32<K>(w, K * c);
        g[c] = (r >> 16) * kLcgMul + kAdd;
        g[c + D] = (r & 0xFFFFu) * kLcgMul + kAdd;
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < 32; ++c) g[c] = pair_state<K>(w, c) * kLcgMul + kAdd;
  }
}

// Sub-units are 4*TPL tiles of one tile row, lane 8*jt + p taking tiles
// J0 + jt + 4t (t < TPL) and rows 2p, 2p+1 of each.

// The layer of sub-unit u of a group: the last whose first sub-unit is <= u.
__device__ __forceinline__ int group_layer_of(const GroupArgs& g, int u) {
  int li = 0, hi = g.count - 1;
  while (li < hi) {
    const int mid = (li + hi + 1) >> 1;
    if (u >= g.l[mid].u_begin) li = mid; else hi = mid - 1;
  }
  return li;
}

// Sub-unit lu of layer a (lane 8*jt + p): decode + MAC of its 4*TPL tiles,
// warp-shuffle reduction, fp32 atomic adds of its 16 row sums.  The first
// call of a warp waits for the preceding grids (x pairs, zeroed row sums)
// after requesting its code words.
template <int K, int CB, int MB, int TPL>
__device__ __forceinline__ void layer_unit(const GroupLayer& a, int lu, int lane, bool& waited) {
  const int jt = lane >> 3;
  const int p = lane & 7;
  constexpr int kTw = RowPair<K>::kTileWords;
  // binary16 of 1024 + the byte-sum centre (1534 for 1MAD, 1150 for mul1)
  const __half2 k1534 = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6400 + byte_sum_centre<CB>())));
  const int nt = a.n / 16;
  const int I = a.row_magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(lu), a.row_magic)) : lu / a.per_row;
  const int J0 = (lu - I * a.per_row) * (4 * TPL) + jt;  // this lane's first tile
  const uint32_t* tp = a.codes + (static_cast<size_t>(I) * nt + J0) * kTw;
  // this lane's words: from word pK of each tile; the last row pair's words
  // past the tile's end wrap to its start (p = 7, words K ..)
  const uint32_t* lp = tp + p * K;
  const uint32_t* lw = lp - (p == 7 ? kTw : 0);
  constexpr int kPw = RowPair<K>::kPairWords;
  auto load_pair = [&](int toff, uint32_t (&wd)[kPw]) {
#pragma unroll
    for (int i = 0; i < kPw; ++i) wd[i] = __ldg((i < K ? lp : lw) + toff + i);
  };

  // Code words two tiles ahead of their decode.
  uint32_t w[2][kPw];
  if (J0 < nt) load_pair(0, w[0]);
  if (TPL > 1 && J0 + 4 < nt) load_pair(4 * kTw, w[1]);
  // The x pairs and the zeroed row sums come from the preceding grids on
  // the stream; the code words above do not.
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
      const uint4* xrow = reinterpret_cast<const uint4*>(a.xdup + static_cast<size_t>(J) * 16);
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
        for (int b = 0; b < MB; ++b) xv[b] = xrow[static_cast<size_t>(b) * (a.n / 4) + q];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * q + j;
          if constexpr (!byte_sum_code<CB>()) {
            const uint32_t pa = mask_xor_3inst(gen[c]);
            const uint32_t pb = mask_xor_3inst(gen[16 + c]);
#pragma unroll
            for (int b = 0; b < MB; ++b) {
              const uint32_t xw = j == 0 ? xv[b].x : j == 1 ? xv[b].y : j == 2 ? xv[b].z : xv[b].w;
              const __half2 x2 = *reinterpret_cast<const __half2*>(&xw);
              ha[b] = __hfma2(*reinterpret_cast<const __half2*>(&pa), x2, ha[b]);
              hb[b] = __hfma2(*reinterpret_cast<const __half2*>(&pb), x2, hb[b]);
            }
          } else {
            const uint32_t ra = __dp4a(summed_bytes<CB>(gen[c]), 0x01010101u, 0x6400u);
            const uint32_t rb2 = __dp4a(summed_bytes<CB>(gen[16 + c]), 0x01010101u, 0x6400u);
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
        if constexpr (!byte_sum_code<CB>()) {
          acc[b][0] += __low2float(ha[b]) + __high2float(ha[b]);
          acc[b][1] += __low2float(hb[b]) + __high2float(hb[b]);
        } else {
          acc[b][0] += __low2float(ha[b]);
          acc[b][1] += __high2float(ha[b]);
        }
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
      float* z = a.zacc + static_cast<size_t>(b) * a.m + I * 16 + 2 * p;
      atomicAdd(z, acc[b][0]);
      atomicAdd(z + 1, acc[b][1]);
    }
  }
}

// Warp w of CTA b takes the sub-units w * grid + b + i * (grid * warps).
// (A device-wide atomic counter cost more than it saved: one L2 address taking
// an atomic from every warp per sub-unit.)
template <int K, int CB, int MB, int TPL>
__device__ __forceinline__ void layer_body(const GroupArgs& g) {
  constexpr int kWarps = layer_warps<MB>();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int stride = static_cast<int>(gridDim.x) * kWarps;
  // The output kernel may be scheduled now (it waits for this grid to finish).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  bool waited = false;
  // CTA-fastest numbering: the sub-units of the last partial round (one more
  // for some warps) fall on every SM alike, not on the first CTAs only.
  int u = warp * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
  if (u >= g.units) return;
  int li = group_layer_of(g, u);
  for (; u < g.units; u += stride) {
    // a warp's sub-units increase, so its layer index only moves forward
    while (li + 1 < g.count && u >= g.l[li + 1].u_begin) ++li;
    const GroupLayer& a = g.l[li];
    layer_unit<K, CB, MB, TPL>(a, u - a.u_begin, lane, waited);
  }
}

template <int K, int CB, int MB, int TPL>
__global__ void __maxnreg__(layer_max_regs<K>()) layer_kernel(const GroupArgs g) {
  layer_body<K, CB, MB, TPL>(g);
}

template <int K, int CB, int MB, int TPL>
__global__ void __launch_bounds__(32 * layer_warps<MB>(), 1) layer_kernel_wide(const GroupArgs g) {
  layer_body<K, CB, MB, TPL>(g);
}

// The sub-units of code CB (up to `end`) of a one-K kernel, continuing the
// warp's sequence u; returns where it stopped.
template <int K, int CB>
__device__ __forceinline__ int kset_loop(const GroupArgs& g, int u, int stride, int end, int& li, int lane,
                                         bool& waited) {
  for (; u < end; u += stride) {
    while (li + 1 < g.count && u >= g.l[li + 1].u_begin) ++li;
    const GroupLayer& a = g.l[li];
    layer_unit<K, CB, 1, 8>(a, u - a.u_begin, lane, waited);
  }
  return u;
}

// Batch 1, 32-tile sub-units: the layers of all four codes of one K, ordered
// by code, in one launch.  A warp's sub-units (numbered and interleaved as in
// layer_body) run through four loops in turn, one per code, each with its own
// decode inlined, so that the step's layers of one K share one launch ramp
// and one tail.
template <int K>
__global__ void __maxnreg__(layer_max_regs<K>()) layer_kernel_kset(const GroupArgs g) {
  constexpr int kWarps = layer_warps<1>();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int stride = static_cast<int>(gridDim.x) * kWarps;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  bool waited = false;
  int u = warp * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
  if (u >= g.units) return;
  int li = group_layer_of(g, u);
  u = kset_loop<K, kCb3Inst>(g, u, stride, g.code_end[0], li, lane, waited);
  u = kset_loop<K, kCb1Mad>(g, u, stride, g.code_end[1], li, lane, waited);
  u = kset_loop<K, kCbMcg>(g, u, stride, g.code_end[2], li, lane, waited);
  kset_loop<K, kCbMul1>(g, u, stride, g.code_end[3], li, lane, waited);
}

template <int K>
exl3_status launch_kset_t(const GroupArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.ctas));
  cfg.blockDim = dim3(32 * layer_warps<1>());
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, layer_kernel_kset<K>, a) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

template <int K, int CB, int MB, int TPL>
exl3_status launch_layer_t(const GroupArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.ctas));
  cfg.blockDim = dim3(32 * layer_warps<MB>());
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if constexpr (MB == 1)
    e = cudaLaunchKernelEx(&cfg, layer_kernel<K, CB, MB, TPL>, a);
  else
    e = cudaLaunchKernelEx(&cfg, layer_kernel_wide<K, CB, MB, TPL>, a);
  if (e != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

template <int K, int CB, int MB>
exl3_status launch_seg_layer_t(const LayerArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.ctas));
  cfg.blockDim = dim3(kSegThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, seg_layer_kernel<K, CB, MB>, a) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

// The segment kernel (batch chunks of 1 or 2).
template <int K, int CB>
exl3_status launch_seg_cb(const LayerArgs& a, int mb, cudaStream_t stream) {
  switch (mb) {
    case 1: return launch_seg_layer_t<K, CB, 1>(a, stream);
    case 2: return launch_seg_layer_t<K, CB, 2>(a, stream);
    default: return EXL3_ERR_BATCH;
  }
}

// The sub-unit kernel over a group of layers (sub-units of a.sub = 32, 16, 8
// or 4 tiles: 8, 4, 2 or 1 tiles per lane; 32 at batch 1 only).
template <int K, int CB, int MB>
exl3_status launch_group_mb(const GroupArgs& a, cudaStream_t stream) {
  switch (a.sub) {
    case 32:
      if constexpr (MB == 1) return launch_layer_t<K, CB, MB, 8>(a, stream);
      return EXL3_ERR_BATCH;
    case 16: return launch_layer_t<K, CB, MB, 4>(a, stream);
    case 8: return launch_layer_t<K, CB, MB, 2>(a, stream);
    default: return launch_layer_t<K, CB, MB, 1>(a, stream);
  }
}

template <int K, int CB>
exl3_status launch_group_cb(const GroupArgs& a, int mb, cudaStream_t stream) {
  switch (mb) {
    case 1: return launch_group_mb<K, CB, 1>(a, stream);
    case 2: return launch_group_mb<K, CB, 2>(a, stream);
    case 4: return launch_group_mb<K, CB, 4>(a, stream);
    case 8: return launch_group_mb<K, CB, 8>(a, stream);
    default: return EXL3_ERR_BATCH;
  }
}

template <int K>
exl3_status launch_layer_dispatch(const LayerArgs& a, int mb, cudaStream_t stream) {
  switch (a.codebook) {
    case kCb3Inst: return launch_seg_cb<K, kCb3Inst>(a, mb, stream);
    case kCb1Mad: return launch_seg_cb<K, kCb1Mad>(a, mb, stream);
    case kCbMcg: return launch_seg_cb<K, kCbMcg>(a, mb, stream);
    default: return launch_seg_cb<K, kCbMul1>(a, mb, stream);
  }
}

template <int K>
exl3_status launch_group_dispatch(const GroupArgs& a, int codebook, int mb, cudaStream_t stream) {
  switch (codebook) {
    case kCb3Inst: return launch_group_cb<K, kCb3Inst>(a, mb, stream);
    case kCb1Mad: return launch_group_cb<K, kCb1Mad>(a, mb, stream);
    case kCbMcg: return launch_group_cb<K, kCbMcg>(a, mb, stream);
    default: return launch_group_cb<K, kCbMul1>(a, mb, stream);
  }
}

}  // namespace exl3

#define EXL3_DEFINE_LAYER_LAUNCHER(KK)                                                         \
  namespace exl3 {                                                                             \
  exl3_status launch_layer_k##KK(const LayerArgs& a, int mb, cudaStream_t stream) {            \
    return launch_layer_dispatch<KK>(a, mb, stream);                                           \
  }                                                                                            \
  exl3_status launch_group_k##KK(const GroupArgs& a, int codebook, int mb, cudaStream_t stream) { \
    return launch_group_dispatch<KK>(a, codebook, mb, stream);                                 \
  }                                                                                            \
  exl3_status launch_group_kset_k##KK(const GroupArgs& a, cudaStream_t stream) {               \
    return launch_kset_t<KK>(a, stream);                                                       \
  }                                                                                            \
  }
