// Fused layer kernel, tensor-core path (tcgen05, sm_103a):
//   y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x))))   for 1 <= M <= 32.
//
// The decoded 16x16 tiles feed tcgen05 MMAs directly from tensor memory:
//
//  * Operand A (128 weight rows x K) lives in TMEM.  Each decode thread owns one
//    weight row of the CTA's 128-row block (TMEM lane = row) and, per pipeline
//    stage, decodes 32 consecutive weights of that row (one row of two
//    adjacent 16x16 tiles), writing one 32-bit TMEM column per weight with
//    tcgen05.st.  The 32-bit column holds a pair of binary16 values whose sum
//    is the weight: for 3INST the two halves straight out of the mask/XOR step
//    ("Trellis Quantization" Part nine), for 1MAD the half 1024 + S (the dp4a
//    byte sum spliced into the mantissa of 1024, the int-to-half trick of Part
//    three) and +0.  So the MMA's K dimension is twice the weight count.
//  * Operand B (K x N, N = batch padded to 16 or 32) is the rotated x slice in
//    shared memory, each value duplicated along K to match the pairs, in the
//    canonical K-major no-swizzle layout (8x16-byte core matrices).
//  * D (128 x N fp32) accumulates in TMEM; the epilogue reads it with
//    tcgen05.ld.  For 1MAD, D = sum (1024 + S) x, so z = C (D - 1534 sum x).
//
// Roles: warps 0-7 decode (two warpgroups take alternate stages; a warp may
// only touch its own 32-lane quarter of TMEM, warps w and w+4 share one),
// warp 8 allocates TMEM and one of its lanes issues the MMAs and commits.
// Synchronization: per A slot a "full" mbarrier (128 decode-thread arrivals)
// and an "empty" mbarrier (tcgen05.commit), plus a "done" mbarrier after the
// last MMA.  Every wait is bounded: on timeout the thread sets an error bit in
// the status word, the CTA skips the rest of its work, waits (bounded) for its
// own MMAs, frees its TMEM and exits.
//
// Split-K and the output transform reuse the scheme of the warp-shuffle path:
// fp32 partial sums + an atomic ticket, the last CTA of a row block finishes.
#pragma once

#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {
namespace tc {

constexpr int kDecodeWarps = 8;
constexpr int kThreads = (kDecodeWarps + 1) * 32;
constexpr int kSlots = 4;            // A stages in TMEM
constexpr int kStageCols = 32;       // weights per row per stage (two tiles)
constexpr int kTmemCols = 256;       // D (<= 32) + 4 x 32 A columns, power of 2
constexpr int kDCol = 0;
constexpr int kACol = 32;
constexpr uint32_t kSpinLimit = 1u << 20;  // about a second of try_wait polling

// ---- PTX wrappers ---------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] x B[smem desc], kind::f16, cta_group::1.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, canonical K-major layout without swizzle:
// start address, leading-dimension byte offset (between the two core matrices
// of a 16-element K step), stride byte offset (between 8-row groups along N),
// descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: D fp32, A and B fp16, both K-major,
// M = 128, N = NB.
template <int NB>
__host__ __device__ constexpr uint32_t idesc_f16() {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(NB >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

// ---- decode of one row's 32 weights of a stage -------------------------------

// Words covering bits [0, 15K + 16) of one 16-step tile row after the row's
// start offset (0 or 16 bits) has been removed.
template <int K>
struct RowWords {
  static constexpr int kTileWords = 8 * K;
  static constexpr int kRaw = (16 + 15 * K + 16 + 31) / 32;  // with a possible 16-bit offset
  static constexpr int kAligned = (15 * K + 16 + 31) / 32;
};

// Load the words of tile row rr (0..15) of one tile, circularly.
template <int K>
__device__ __forceinline__ void load_tile_row(const uint32_t* __restrict__ tile, int q0,
                                              uint32_t (&raw)[RowWords<K>::kRaw]) {
#pragma unroll
  for (int i = 0; i < RowWords<K>::kRaw; ++i) {
    int idx = q0 + i;
    if (idx >= RowWords<K>::kTileWords) idx -= RowWords<K>::kTileWords;
    raw[i] = __ldg(tile + idx);
  }
}

// State of step c (0..15) of a tile row from left-aligned words.
template <int K>
__device__ __forceinline__ uint32_t row_bits32(const uint32_t (&w)[RowWords<K>::kAligned + 1], int b) {
  const int q = b >> 5;
  const int sh = b & 31;
  return sh == 0 ? w[q] : __funnelshift_l(w[q + 1], w[q], sh);
}

template <int K>
__device__ __forceinline__ void row_states(const uint32_t (&raw)[RowWords<K>::kRaw], uint32_t off,
                                           uint32_t (&s)[16]) {
  uint32_t w[RowWords<K>::kAligned + 1];
#pragma unroll
  for (int i = 0; i <= RowWords<K>::kAligned; ++i) {
    if constexpr (K % 2 == 0) {
      w[i] = i < RowWords<K>::kRaw ? raw[i] : 0u;  // rows of even K start word-aligned
    } else {
      const uint32_t lo = i + 1 < RowWords<K>::kRaw ? raw[i + 1] : 0u;
      w[i] = i < RowWords<K>::kRaw ? __funnelshift_l(lo, raw[i], off) : 0u;
    }
  }
  if constexpr (16 % K == 0 && K > 1) {
    constexpr int D = 16 / K;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      if ((c / D) % 2 == 0) {
        const uint32_t r = row_bits32<K>(w, K * c);
        s[c] = r >> 16;
        s[c + D] = r & 0xFFFFu;
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) s[c] = row_bits32<K>(w, K * c) >> 16;
  }
}

// 32-bit TMEM column of one weight: a pair of binary16 values summing to it
// (the 1MAD value is offset by 1534 and unscaled; the epilogue corrects).
template <int CB>
__device__ __forceinline__ uint32_t pair_code(uint32_t s) {
  const uint32_t x = lcg(s);
  if constexpr (CB == kCb3Inst) {
    return (x & k3InstMask) ^ k3InstMagic;
  } else {
    return __dp4a(x, 0x01010101u, 0x6400u);  // binary16 bits of 1024 + S, high half +0
  }
}

struct TcShared {
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  uint64_t done;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t ticket;
  float xsum[32];  // per batch row: sum of the binary16 x-tilde values of the slice
  float zs[32 * 128];
};

template <int K, int CB, int NB>
__global__ void __launch_bounds__(kThreads, 1) tc_layer_kernel(LayerArgs a, int M) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  TcShared& sh = *reinterpret_cast<TcShared*>(smem_raw);
  // B operand after the control block, 1024-byte aligned.
  unsigned char* bsm = smem_raw + ((sizeof(TcShared) + 1023) & ~static_cast<size_t>(1023));

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
  const int nstages = ns / kStageCols;

  // ---- set-up ---------------------------------------------------------------
  if (warp == kDecodeWarps) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
  }
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sh.full[i], 128);
      mbar_init(&sh.empty[i], 1);
    }
    mbar_init(&sh.done, 1);
    sh.abort = 0;
  }
  if (tid < 32) sh.xsum[tid] = 0.f;
  __syncthreads();

  // B operand: element (n, k) of the N x 2ns K-major matrix at core matrix
  // (k / 8, n / 8), offset ((k/8) * (NB/8) + n/8) * 128 + (n % 8) * 16 + (k % 8) * 2.
  // Rows n >= M are zero.  Each value of x-tilde is stored twice (k = 2c, 2c+1).
  {
    const int nkb = ns / kRowBlock;
    for (int job = warp; job < NB * nkb; job += kThreads / 32) {
      const int n = job / nkb;
      const int kb = job - n * nkb;
      const int col = c0 + kb * kRowBlock + 4 * lane;   // 4 x values -> k = 8j .. 8j+7
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (n < M) {
        const uint2 xr = *reinterpret_cast<const uint2*>(a.x + static_cast<size_t>(n) * a.n + col);
        const __half2 x01 = *reinterpret_cast<const __half2*>(&xr.x);
        const __half2 x23 = *reinterpret_cast<const __half2*>(&xr.y);
        v[0] = __low2float(x01);
        v[1] = __high2float(x01);
        v[2] = __low2float(x23);
        v[3] = __high2float(x23);
        if (a.s_in != nullptr) {
          const uint2 sr = *reinterpret_cast<const uint2*>(a.s_in + col);
          const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
          const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
          v[0] *= __low2float(s01);
          v[1] *= __high2float(s01);
          v[2] *= __low2float(s23);
          v[3] *= __high2float(s23);
          fwht128_warp(v, lane);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
        }
      }
      __half h[4];
      float hs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        h[j] = __float2half_rn(v[j]);
        hs += __half2float(h[j]);
      }
      const int kc = (kb * kRowBlock + 4 * lane) / 4;  // core-matrix column: k / 8 with k = 2 * (local col)
      const uint32_t off = (static_cast<uint32_t>(kc) * (NB / 8) + n / 8) * 128u + (n % 8) * 16u;
      uint4 pk;
      pk.x = static_cast<uint32_t>(__half_as_ushort(h[0])) * 0x10001u;
      pk.y = static_cast<uint32_t>(__half_as_ushort(h[1])) * 0x10001u;
      pk.z = static_cast<uint32_t>(__half_as_ushort(h[2])) * 0x10001u;
      pk.w = static_cast<uint32_t>(__half_as_ushort(h[3])) * 0x10001u;
      *reinterpret_cast<uint4*>(bsm + off) = pk;
      if (CB == kCb1Mad && n < M) {
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) hs += __shfl_xor_sync(0xFFFFFFFFu, hs, d);
        if (lane == 0) atomicAdd(&sh.xsum[n], hs);
      }
    }
  }
  // Generic-proxy writes of B must be visible to the tensor core (async proxy).
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp < kDecodeWarps) {
    // ---- decode producers ---------------------------------------------------
    const int g = warp >> 2;              // warpgroup: stages s with s % 2 == g
    const int quarter = warp & 3;         // TMEM lanes 32*quarter ..
    const int row = quarter * 32 + lane;  // row of the 128-row block
    const int I = rb * 8 + (row >> 4);
    const int rr = row & 15;
    const int q0 = (rr * K) >> 1;
    const uint32_t off = static_cast<uint32_t>((rr * K) & 1) * 16u;
    const int tiles_per_row = a.n / 16;
    const uint32_t* rowp = a.codes + (static_cast<size_t>(I) * tiles_per_row + c0 / 16) * (8 * K);
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);

    uint32_t raw0[RowWords<K>::kRaw], raw1[RowWords<K>::kRaw];
    int s = g;
    if (s < nstages) {
      load_tile_row<K>(rowp + static_cast<size_t>(2 * s) * 8 * K, q0, raw0);
      load_tile_row<K>(rowp + static_cast<size_t>(2 * s + 1) * 8 * K, q0, raw1);
    }
    for (; s < nstages; s += 2) {
      uint32_t st0[16], st1[16];
      row_states<K>(raw0, off, st0);
      row_states<K>(raw1, off, st1);
      if (s + 2 < nstages) {  // prefetch the next stage of this warpgroup
        load_tile_row<K>(rowp + static_cast<size_t>(2 * (s + 2)) * 8 * K, q0, raw0);
        load_tile_row<K>(rowp + static_cast<size_t>(2 * (s + 2) + 1) * 8 * K, q0, raw1);
      }
      uint32_t v[32];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        v[c] = pair_code<CB>(st0[c]);
        v[16 + c] = pair_code<CB>(st1[c]);
      }
      const int slot = s % kSlots;
      const int use = s / kSlots;
      bool ok = true;
      if (use > 0) ok = mbar_wait(&sh.empty[slot], (use - 1) & 1);
      if (!ok) atomicOr(&sh.abort, 1u);
      // warp-uniform exit: tcgen05.st below is a whole-warp instruction
      if (__any_sync(0xFFFFFFFFu, !ok || *reinterpret_cast<volatile uint32_t*>(&sh.abort) != 0u)) break;
      tmem_st32(lane_addr + kACol + slot * kStageCols, v);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sh.full[slot]);
    }
  } else if (lane == 0) {
    // ---- MMA issuer -------------------------------------------------------
    constexpr uint32_t idesc = idesc_f16<NB>();
    const uint32_t bbase = smem_u32(bsm);
    constexpr uint32_t kLbo = (NB / 8) * 128;  // next 8 K-elements
    constexpr uint32_t kSbo = 128;             // next 8 rows of N
    for (int s = 0; s < nstages; ++s) {
      const int slot = s % kSlots;
      if (!mbar_wait(&sh.full[slot], (s / kSlots) & 1)) {
        atomicOr(&sh.abort, 1u);
        break;
      }
      if (*reinterpret_cast<volatile uint32_t*>(&sh.abort)) break;
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t kk = static_cast<uint32_t>(s) * 64u + 16u * j;  // K offset (halves)
        const uint64_t bd = smem_desc(bbase + (kk / 8) * kLbo, kLbo, kSbo);
        mma_f16_ts(tmem + kDCol, tmem + kACol + slot * kStageCols + 8 * j, bd, idesc,
                   (s > 0 || j > 0) ? 1u : 0u);
      }
      mma_commit(&sh.empty[slot]);
    }
    mma_commit(&sh.done);
  }

  // ---- epilogue: D -> row sums ---------------------------------------------
  __syncwarp();
  const bool ok_done = mbar_wait(&sh.done, 0);
  if (!ok_done) atomicOr(&sh.abort, 1u);
  tc_fence_after();
  if (warp < 4) {
    const int row = warp * 32 + lane;
    float d[16];
    tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kDCol, d);
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      if (n < M) {
        float z = d[n];
        if (CB == kCb1Mad) z = (z - 1534.0f * sh.xsum[n]) * kOneMadScale;
        sh.zs[n * kRowBlock + row] = z;
      }
    }
    if constexpr (NB == 32) {
      tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kDCol + 16, d);
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        if (16 + n < M) {
          float z = d[n];
          if (CB == kCb1Mad) z = (z - 1534.0f * sh.xsum[16 + n]) * kOneMadScale;
          sh.zs[(16 + n) * kRowBlock + row] = z;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kDecodeWarps) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (sh.abort) {
    if (tid == 0 && a.status != nullptr) atomicOr(a.status, 1u);
    return;
  }

  // ---- split-K combine -------------------------------------------------------
  if (a.splits > 1) {
    float* part = a.partials + static_cast<size_t>(split) * M * a.m;
    for (int i = tid; i < M * kRowBlock; i += kThreads) {
      const int b = i / kRowBlock;
      const int r = i - b * kRowBlock;
      part[static_cast<size_t>(b) * a.m + rb * kRowBlock + r] = sh.zs[i];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) sh.ticket = atomicAdd(a.counters + rb, 1u);
    __syncthreads();
    if (sh.ticket != static_cast<uint32_t>(a.splits - 1)) return;
    __threadfence();
    for (int i = tid; i < M * kRowBlock; i += kThreads) {
      const int b = i / kRowBlock;
      const int r = i - b * kRowBlock;
      float acc = 0.f;
      for (int sp = 0; sp < a.splits; ++sp)
        acc += __ldcg(a.partials + (static_cast<size_t>(sp) * M + b) * a.m + rb * kRowBlock + r);
      sh.zs[i] = acc;
    }
    if (tid == 0) a.counters[rb] = 0u;
    __syncthreads();
  }

  // ---- scale, output signs + FWHT, binary16 ------------------------------------
  for (int b = warp; b < M; b += kThreads / 32) {
    const int r0 = rb * kRowBlock + 4 * lane;
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = sh.zs[b * kRowBlock + 4 * lane + j];
    {
      const uint2 sr = *reinterpret_cast<const uint2*>(a.scales + r0);
      const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
      const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
      v[0] *= __low2float(s01);
      v[1] *= __high2float(s01);
      v[2] *= __low2float(s23);
      v[3] *= __high2float(s23);
    }
    if (a.s_out != nullptr) {
      const uint2 sr = *reinterpret_cast<const uint2*>(a.s_out + r0);
      const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
      const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
      v[0] *= __low2float(s01);
      v[1] *= __high2float(s01);
      v[2] *= __low2float(s23);
      v[3] *= __high2float(s23);
      fwht128_warp(v, lane);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
    }
    const __half2 o01 = __floats2half2_rn(v[0], v[1]);
    const __half2 o23 = __floats2half2_rn(v[2], v[3]);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&o01);
    o.y = *reinterpret_cast<const uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(a.y + static_cast<size_t>(b) * a.m + r0) = o;
  }
}

// Shared memory: control block + B operand (NB x 2ns halves).
inline size_t tc_smem_bytes(int nb, int ns) {
  const size_t ctrl = (sizeof(TcShared) + 1023) & ~static_cast<size_t>(1023);
  return ctrl + static_cast<size_t>(nb) * 2 * ns * sizeof(__half);
}

template <int K, int CB, int NB>
exl3_status launch_tc_t(const LayerArgs& a, int M, cudaStream_t stream) {
  const int nblk = a.n / kRowBlock;
  const int ns_max = ((nblk + a.splits - 1) / a.splits) * kRowBlock;
  // At least 100 KB so that no more than two CTAs are resident per SM: two
  // 256-column TMEM allocations fill the SM's 512 columns exactly, and a third
  // CTA would have to wait in tcgen05.alloc.
  size_t smem = tc_smem_bytes(NB, ns_max);
  if (smem < 100 * 1024) smem = 100 * 1024;
  if (cudaFuncSetAttribute(tc_layer_kernel<K, CB, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return EXL3_ERR_CUDA;
  const dim3 grid(a.m / kRowBlock, a.splits);
  tc_layer_kernel<K, CB, NB><<<grid, kThreads, smem, stream>>>(a, M);
  return launch_status();
}

template <int K>
exl3_status launch_tc_dispatch(const LayerArgs& a, int M, cudaStream_t stream) {
  if (a.codebook == kCb3Inst)
    return M <= 16 ? launch_tc_t<K, kCb3Inst, 16>(a, M, stream) : launch_tc_t<K, kCb3Inst, 32>(a, M, stream);
  return M <= 16 ? launch_tc_t<K, kCb1Mad, 16>(a, M, stream) : launch_tc_t<K, kCb1Mad, 32>(a, M, stream);
}

}  // namespace tc
}  // namespace exl3

#define EXL3_DEFINE_TC_LAUNCHER(KK)                                                        \
  namespace exl3 {                                                                         \
  exl3_status launch_tc_k##KK(const LayerArgs& a, int M, cudaStream_t stream) {            \
    return tc::launch_tc_dispatch<KK>(a, M, stream);                                       \
  }                                                                                        \
  }
