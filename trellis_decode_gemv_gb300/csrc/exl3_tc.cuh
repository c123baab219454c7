// Fused layer kernel, tensor-core path (tcgen05, sm_103a):
//   z = W-hat x-tilde   for 1 <= M <= 32 batch rows,
// accumulated in fp32 into the workspace row sums; the input transform
// (x-tilde = Hb(s_in (.) x), laid out as operand B) runs before it and the
// output transform (y = Hb(s_out (.) (scale (.) z))) after it, both chained by
// programmatic dependent launch.
//
// The decoded 16x16 tiles feed tcgen05 MMAs directly from tensor memory:
//
//  * Operand A (128 weight rows x 128) lives in TMEM.  Each decode thread owns
//    one weight row of a 128-row block (TMEM lane = row) and, per 128-column
//    chunk, decodes 32 consecutive weights of that row (one row of two
//    adjacent 16x16 tiles), writing two binary16 weights per 32-bit TMEM
//    column with tcgen05.st (the lower half holds the even K element).  3INST
//    weights are the binary16 sums of the two halves of the mask/XOR step
//    ("Trellis Quantization" Part nine), formed for two columns at once by two
//    byte permutes and one packed add -- exactly the defined binary16
//    weights; 1MAD weights are stored as the half 1024 + S (the dp4a byte sum
//    spliced into the mantissa of 1024, the int-to-half trick of Part three),
//    paired by one byte permute.
//  * Operand B (128 x N, N = batch padded to 16 or 32) is the chunk's slice of
//    x-tilde, binary16, in the canonical K-major no-swizzle layout (8x16-byte
//    core matrices), fetched as one contiguous bulk copy per chunk.
//  * D (128 x N fp32) accumulates in TMEM over a run of chunks of one 128-row
//    block.  For 1MAD, D = sum (1024 + S) x, so z = C (D - 1534 sum x) with
//    C = 1/sqrt(21845); the sums of x per 128 block come with operand B.
//
// Persistent kernel, one CTA per SM, stream-K work split: the (m/128) x
// (n/128) chunks, row-block major, are cut into gridDim.x contiguous ranges;
// the chunks of one range that share a row block form a run, whose D the
// epilogue adds into the row sums with fp32 reductions.  Warp roles:
//   warps 0-15  decode: four warpgroups; warpgroup g decodes tile columns
//               2g, 2g+1 of every chunk (a warp only reaches its own 32-lane
//               quarter of TMEM, so the four warps of a warpgroup cover the
//               128 rows);
//   warps 16-19 epilogue: tcgen05.ld of each run's D, 1MAD correction,
//               reduction into the row sums;
//   warp 20     MMA issue (one lane, 8 MMAs of 128 x N x 16 per chunk) and
//               TMEM allocation;
//   warp 21     code producer: 1-D bulk copies (cp.async.bulk) of each
//               chunk's eight tile-row strips of packed codes (one lane per
//               strip) into a 4- or 8-deep shared-memory ring;
//   warp 22     operand-B producer: waits for the preceding transform kernel,
//               then one bulk copy per chunk into a ring slot paired with the
//               chunk's TMEM slot.
// mbarriers: code ring full/empty, A full/empty and B full (6 chunk slots),
// D full/empty (2 TMEM accumulators).  Every wait is bounded: on timeout the
// thread sets the CTA's abort flag and the workspace status word, every role
// stops, the producers wait (bounded) for their copies in flight, the MMA lane
// for its MMAs, TMEM is freed and the CTA exits.
#pragma once

#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {
namespace tc {

constexpr int kDecodeWarps = 16;
constexpr int kEpiWarp0 = 16;
constexpr int kMmaWarp = 20;
constexpr int kTmaWarp = 21;
constexpr int kBWarp = 22;
constexpr int kThreads = 23 * 32;
constexpr int kMaxRing = 8;
constexpr int kMaxSlots = 4;
constexpr int kMaxNB = 128;
constexpr int kTmemCols = 512;
constexpr int kDCol = 0;                // D buffers at columns 0 and Cfg::kDStride
constexpr int kRowPadWords = 16;        // keeps tile-row strips 64 B apart from a bank multiple

// Layout of the kernel for K-bit codes and N = NB batch columns.
//  NB <= 32 (skinny batches): chunks of 16 tile columns (256 input columns)
//    when n allows it, else 8; 3 A slots of 128 TMEM columns after D at
//    columns 0 and 32; 8 code chunks in flight for K <= 4, 4 above; D is
//    transposed through shared memory for 16-byte reductions.
//  NB = 128 (prefill passes of 128 batch rows): chunks of 8 tile columns;
//    4 A slots of 64 columns after D at columns 0 and 128; 4 code chunks in
//    flight; 32 KB operand-B slots; D transposed 16 batch columns at a time.
template <int K, int NB>
struct TcCfg {
  static constexpr bool kWide = NB > 32;
  static constexpr int kMaxTiles = kWide ? 8 : 16;
  static constexpr int kSlots = kWide ? 4 : 3;
  static constexpr int kSlotCols = kWide ? 64 : 128;
  static constexpr int kDStride = kWide ? NB : 32;
  static constexpr int kACol = 2 * kDStride;
  static constexpr int kRing = kWide ? 4 : (K <= 4 ? 8 : 4);
  static constexpr int kRowWords = kMaxTiles * 8 * K + kRowPadWords;
  static constexpr int kChunkBytes = 8 * kRowWords * 4;
  static constexpr int kBSlotBytes = NB * kMaxTiles * 16 * 2;
  // D transposed to [batch][row] for 16-byte reductions: every batch column
  // (skinny), or 16 at a time (wide)
  static constexpr int kTransposeCols = kWide ? 16 : 32;
  static constexpr int kTransposeBytes = kTransposeCols * 128 * 4;
  static_assert(kACol + kSlots * kSlotCols <= kTmemCols, "TMEM columns");
  static_assert(kSlots <= kMaxSlots && kRing <= kMaxRing && NB <= kMaxNB, "barrier arrays");
};
constexpr uint32_t kSpinLimit = 1u << 20;  // about a second of try_wait polling
constexpr int kEpiBarrier = 1;          // named barrier of the epilogue warps

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

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// Bounded wait for the phase with the given parity to complete.
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

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
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

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
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

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarrier), "n"(128) : "memory");
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

// ---- decode of one tile row ---------------------------------------------------

template <int K>
struct RowWords {
  static constexpr int kTileWords = 8 * K;
  static constexpr int kRaw = (16 + 15 * K + 16 + 31) / 32;  // with a possible 16-bit offset
  static constexpr int kAligned = (15 * K + 16 + 31) / 32;
};

template <int K>
__device__ __forceinline__ uint32_t row_bits32(const uint32_t (&w)[RowWords<K>::kAligned + 1], int b) {
  const int q = b >> 5;
  const int sh = b & 31;
  return sh == 0 ? w[q] : __funnelshift_l(w[q + 1], w[q], sh);
}

// The 16 states of one tile row from its raw words; `off` (0 or 16) is the bit
// offset of the row's first window inside raw[0].
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

// One 32-bit TMEM column: the binary16 values of two consecutive weights of a
// row, the first in the lower half (the 1MAD values are offset by 1534 and
// unscaled; the epilogue corrects).
template <int CB>
__device__ __forceinline__ uint32_t pack_two(uint32_t s0, uint32_t s1) {
  const uint32_t x0 = generate<CB>(s0);
  const uint32_t x1 = generate<CB>(s1);
  if constexpr (!byte_sum_code<CB>()) {
    const uint32_t h0 = mask_xor_3inst(x0);
    const uint32_t h1 = mask_xor_3inst(x1);
    const uint32_t lo = __byte_perm(h0, h1, 0x5410);  // (lo half of w0, lo half of w1)
    const uint32_t hi = __byte_perm(h0, h1, 0x7632);  // (hi half of w0, hi half of w1)
    const __half2 w = __hadd2(*reinterpret_cast<const __half2*>(&lo), *reinterpret_cast<const __half2*>(&hi));
    return *reinterpret_cast<const uint32_t*>(&w);
  } else {
    const uint32_t d0 = __dp4a(summed_bytes<CB>(x0), 0x01010101u, 0x6400u);  // binary16 bits of 1024 + S
    const uint32_t d1 = __dp4a(summed_bytes<CB>(x1), 0x01010101u, 0x6400u);
    return __byte_perm(d0, d1, 0x5410);
  }
}

// The 32 TMEM column words of two adjacent tiles of one row (raw words as
// loaded for that row of each tile).
template <int K, int CB>
__device__ __forceinline__ void decode_tile_pair(const uint32_t (&raw0)[RowWords<K>::kRaw],
                                                 const uint32_t (&raw1)[RowWords<K>::kRaw], uint32_t off,
                                                 uint32_t (&v)[16]) {
  uint32_t st0[16], st1[16];
  row_states<K>(raw0, off, st0);
  row_states<K>(raw1, off, st1);
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    v[j / 2] = pack_two<CB>(st0[j], st0[j + 1]);
    v[8 + j / 2] = pack_two<CB>(st1[j], st1[j + 1]);
  }
}

struct TcParams {
  LayerArgs a;
  const __half* bimg;  // operand-B images, one per 128-column block
  const float* bsum;   // [M][n/128] sums of x-tilde (1MAD), else unused
  int M;
  int ct;              // tile columns per chunk: 16, or 8 when n is an odd multiple of 128
};

struct TcShared {
  uint64_t ring_full[kMaxRing];
  uint64_t ring_empty[kMaxRing];
  uint64_t a_full[kMaxSlots];
  uint64_t a_empty[kMaxSlots];
  uint64_t b_full[kMaxSlots];
  uint64_t d_full[2];
  uint64_t d_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t epi_go;
  float xsum[kMaxNB];
};

__device__ __forceinline__ bool aborted(const TcShared& sh) {
  return *reinterpret_cast<const volatile uint32_t*>(&sh.abort) != 0u;
}

__device__ __forceinline__ void set_abort(TcShared& sh) { atomicOr(&sh.abort, 1u); }

template <int K, int CB, int NB>
__global__ void __launch_bounds__(kThreads, 1) tc_layer_kernel(TcParams p) {
  using Cfg = TcCfg<K, NB>;
  constexpr int kSlots = Cfg::kSlots;
  constexpr int kRing = Cfg::kRing;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  TcShared& sh = *reinterpret_cast<TcShared*>(smem_raw);
  const size_t ctrl = (sizeof(TcShared) + 1023) & ~static_cast<size_t>(1023);
  // D of a run transposed to [batch][row] (skinny batches), 16-byte aligned
  float* zt = reinterpret_cast<float*>(smem_raw + ctrl);
  unsigned char* bring = smem_raw + ctrl + Cfg::kTransposeBytes;
  uint32_t* ring = reinterpret_cast<uint32_t*>(bring + static_cast<size_t>(kSlots) * Cfg::kBSlotBytes);

  // The output kernel may launch now; it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const LayerArgs& a = p.a;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int tiles_per_row = a.n / 16;
  const int ct = p.ct;
  const int nkb = a.n / (16 * ct);                 // chunks per row block
  const uint32_t bbytes = static_cast<uint32_t>(NB) * 16u * ct * 2u;  // operand B of one chunk
  const long long total = static_cast<long long>(a.m / kRowBlock) * nkb;
  const int lo = static_cast<int>(total * blockIdx.x / gridDim.x);
  const int hi = static_cast<int>(total * (blockIdx.x + 1) / gridDim.x);

  // ---- set-up ---------------------------------------------------------------
  // The code producer initialises its ring and issues the first chunks before
  // the block-wide barrier, so that their HBM latency overlaps the TMEM
  // allocation and the initialisation of the other barriers.
  auto issue_chunk = [&](int seq, int c) {
    const int rb = c / nkb;
    const int kb = c - rb * nkb;
    const int slot = seq % kRing;
    // Lanes 0-7 each copy one tile-row strip; lane 0 posts the byte count first.
    if (lane == 0) mbar_arrive_expect_tx(&sh.ring_full[slot], 8u * ct * 32u * K);
    __syncwarp();
    if (lane < 8) {
      uint32_t* dst = ring + static_cast<size_t>(slot) * (Cfg::kChunkBytes / 4);
      const uint32_t* src = a.codes + (static_cast<size_t>(rb * 8 + lane) * tiles_per_row + kb * ct) * (8 * K);
      bulk_g2s(dst + lane * Cfg::kRowWords, src, ct * 32u * K, &sh.ring_full[slot]);
    }
  };
  int pre = 0;
  if (warp == kTmaWarp) {
    if (lane == 0) {
      for (int i = 0; i < kRing; ++i) {
        mbar_init(&sh.ring_full[i], 1);
        mbar_init(&sh.ring_empty[i], kDecodeWarps);  // one elected arrival per decode warp
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    // Two chunks: issuing more would hold the other warps at the barrier.
    pre = min(2, hi - lo);
    for (int s = 0; s < pre; ++s) issue_chunk(s, lo + s);
  }
  if (warp == kMmaWarp) tmem_alloc(&sh.tmem_base, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sh.a_full[i], kDecodeWarps);
      mbar_init(&sh.a_empty[i], 1);
      mbar_init(&sh.b_full[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.d_full[i], 1);
      mbar_init(&sh.d_empty[i], 128);
    }
    mbar_init(&sh.mma_done, 1);
    sh.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kTmaWarp) {
    // ---- code producer: the remaining chunks into the ring ---------------------------
    int seq = pre;
    for (int c = lo + pre; c < hi; ++c, ++seq) {
      const int slot = seq % kRing;
      const int use = seq / kRing;
      bool ok = true;
      if (use > 0) ok = mbar_wait(&sh.ring_empty[slot], (use - 1) & 1);
      if (!ok) set_abort(sh);
      if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) break;
      issue_chunk(seq, c);
    }
    // Wait (bounded) for every copy issued into the ring to land before exit.
    for (int i = 0; i < kRing && i < seq; ++i) {
      const int s = seq - 1 - i;
      mbar_wait(&sh.ring_full[s % kRing], (s / kRing) & 1);
    }
  } else if (warp == kBWarp) {
    // ---- operand-B producer ----------------------------------------------------------
    // With the failure-detection test hook set this warp posts nothing, so the
    // MMA lane's bounded wait for operand B runs out.
    if (lane == 0 && a.debug_stall == 0) {
      // The images are written by the preceding kernel on the stream.
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int seq = 0;
      for (int c = lo; c < hi; ++c, ++seq) {
        const int kb = c % nkb;
        const int slot = seq % kSlots;
        const int use = seq / kSlots;
        if (use > 0 && !mbar_wait(&sh.a_empty[slot], (use - 1) & 1)) set_abort(sh);
        if (aborted(sh)) break;
        mbar_arrive_expect_tx(&sh.b_full[slot], bbytes);
        bulk_g2s(bring + static_cast<size_t>(slot) * Cfg::kBSlotBytes,
                 p.bimg + static_cast<size_t>(kb) * NB * 16 * ct, bbytes, &sh.b_full[slot]);
      }
      for (int i = 0; i < kSlots && i < seq; ++i) {
        const int s = seq - 1 - i;
        mbar_wait(&sh.b_full[s % kSlots], (s / kSlots) & 1);
      }
    }
  } else if (warp < kDecodeWarps) {
    // ---- decode producers of operand A -------------------------------------------
    // Warpgroup g decodes tile columns g * ct/4 .. g * ct/4 + ct/4 - 1 of every
    // chunk, two adjacent tiles (one 16-column TMEM group) at a time.
    const int g = warp >> 2;
    const int quarter = warp & 3;         // TMEM lanes 32 * quarter ..
    const int row = quarter * 32 + lane;  // row within the 128-row block
    const int trow = row >> 4;            // tile row within the block
    const int rr = row & 15;
    const int q0 = (rr * K) >> 1;
    const uint32_t off = static_cast<uint32_t>((rr * K) & 1) * 16u;
    const int t0 = g * (ct / 4);          // first tile column of this warpgroup
    const bool two = ct == 16;            // a second tile pair per chunk
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + Cfg::kACol + 8 * t0;
    int seq = 0;
    for (int c = lo; c < hi; ++c, ++seq) {
      const int slot = seq % kRing;
      bool ok = mbar_wait(&sh.ring_full[slot], (seq / kRing) & 1);
      if (!ok) set_abort(sh);
      if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) break;
      const uint32_t* rw = ring + static_cast<size_t>(slot) * (Cfg::kChunkBytes / 4) +
                           trow * Cfg::kRowWords + t0 * (8 * K);
      uint32_t raw[4][RowWords<K>::kRaw];
#pragma unroll
      for (int i = 0; i < RowWords<K>::kRaw; ++i) {
        int idx = q0 + i;
        if (idx >= 8 * K) idx -= 8 * K;
        raw[0][i] = rw[idx];
        raw[1][i] = rw[8 * K + idx];
        if (two) {
          raw[2][i] = rw[16 * K + idx];
          raw[3][i] = rw[24 * K + idx];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.ring_empty[slot]);
      uint32_t v0[16], v1[16];
      decode_tile_pair<K, CB>(raw[0], raw[1], off, v0);
      if (two) decode_tile_pair<K, CB>(raw[2], raw[3], off, v1);
      const int aslot = seq % kSlots;
      const int use = seq / kSlots;
      ok = true;
      if (use > 0) ok = mbar_wait(&sh.a_empty[aslot], (use - 1) & 1);
      if (!ok) set_abort(sh);
      if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) break;
      tmem_st16(lane_addr + aslot * Cfg::kSlotCols, v0);
      if (two) tmem_st16(lane_addr + aslot * Cfg::kSlotCols + 16, v1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.a_full[aslot]);
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issue ------------------------------------------------------------------
    // The whole warp runs the loop (waits, descriptors: warp-uniform values);
    // lane 0 issues the MMAs and the commits that track them.
    constexpr uint32_t idesc = idesc_f16<NB>();
    constexpr uint32_t kLbo = (NB / 8) * 128;  // next 8 K-elements
    constexpr uint32_t kSbo = 128;             // next 8 rows of N
    const uint64_t bdesc0 = smem_desc(smem_u32(bring), kLbo, kSbo);
    const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
    const bool two_mma = ct == 16;
    int seq = 0;
    int run = 0;
    bool bad = false;
    for (int c = lo; c < hi && !bad; ++run) {
      const int rb = c / nkb;
      const int end = min(hi, (rb + 1) * nkb);
      const int db = run & 1;
      const bool okd = run < 2 || mbar_wait(&sh.d_empty[db], ((run >> 1) - 1) & 1);
      if (__any_sync(0xFFFFFFFFu, !okd)) {
        set_abort(sh);
        break;
      }
      const uint32_t dt = tm + kDCol + Cfg::kDStride * db;
      for (uint32_t acc = 0; c < end; ++c, ++seq, acc = 1) {
        const int slot = seq % kSlots;
        const uint32_t par = (seq / kSlots) & 1;
        const bool ok = mbar_wait(&sh.a_full[slot], par) && mbar_wait(&sh.b_full[slot], par) && !aborted(sh);
        if (__any_sync(0xFFFFFFFFu, !ok)) {
          set_abort(sh);
          bad = true;
          break;
        }
        tc_fence_after();
        // descriptor start address advances by (bytes >> 4) in its low field
        const uint64_t bd = bdesc0 + ((static_cast<uint32_t>(slot) * Cfg::kBSlotBytes) >> 4);
        const uint32_t at = tm + Cfg::kACol + slot * Cfg::kSlotCols;
        if (lane == 0) {
          // one MMA per tile column (K = 16); the first MMA of a run overwrites D
          mma_f16_ts(dt, at, bd, idesc, acc);
#pragma unroll
          for (int j = 1; j < 8; ++j) mma_f16_ts(dt, at + 8 * j, bd + ((2u * j * kLbo) >> 4), idesc, 1u);
          if (two_mma) {
#pragma unroll
            for (int j = 8; j < 16; ++j) mma_f16_ts(dt, at + 8 * j, bd + ((2u * j * kLbo) >> 4), idesc, 1u);
          }
          mma_commit(&sh.a_empty[slot]);
        }
        __syncwarp();
      }
      if (bad) break;
      if (lane == 0) mma_commit(&sh.d_full[db]);
      __syncwarp();
    }
    if (lane == 0) mma_commit(&sh.mma_done);
    __syncwarp();
    mbar_wait(&sh.mma_done, 0);
  } else {
    // ---- epilogue warps: D of each run into the row sums -----------------------------
    // The block sums of x-tilde come from the preceding grid on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int ew = warp - kEpiWarp0;      // 0..3 = TMEM lane quarter
    const int et = tid - kEpiWarp0 * 32;  // 0..127
    int run = 0;
    for (int c = lo; c < hi; ++run) {
      const int rb = c / nkb;
      const int end = min(hi, (rb + 1) * nkb);
      const int kb0 = c - rb * nkb;
      const int kb1 = end - rb * nkb;
      c = end;
      // Uniform go/stop decision for the four epilogue warps: they share named
      // barriers, so they must leave together.
      if (et == 0) sh.epi_go = aborted(sh) ? 0u : 1u;
      epi_sync();
      if (sh.epi_go == 0u) break;
      if constexpr (byte_sum_code<CB>()) {
        // sum of x-tilde over the run's columns, per batch row
        for (int b = ew; b < p.M; b += 4) {
          float s = 0.f;
          const int nblk = a.n / kRowBlock;  // 128-column blocks per row
          for (int kb = kb0 * (ct / 8) + lane; kb < kb1 * (ct / 8); kb += 32)
            s += __ldcg(p.bsum + static_cast<size_t>(b) * nblk + kb);
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, d);
          if (lane == 0) sh.xsum[b] = s;
        }
        epi_sync();
      }
      const int db = run & 1;
      bool ok = !aborted(sh) && mbar_wait(&sh.d_full[db], (run >> 1) & 1);
      if (!ok) set_abort(sh);
      // tcgen05.ld is a whole-warp instruction: skip it warp-uniformly.
      const int row = ew * 32 + lane;
      float* zblk = a.zacc + static_cast<size_t>(rb) * kRowBlock;
      const bool warp_ok = !__any_sync(0xFFFFFFFFu, !ok);
      if (warp_ok) tc_fence_after();
      // D in slices of kTransposeCols batch columns: TMEM -> registers (1MAD
      // and mul1 corrected) -> shared memory [batch][row] -> 16-byte
      // reductions of four consecutive rows of one batch row.
      constexpr int kTc = Cfg::kTransposeCols;
      const int slices = (p.M + kTc - 1) / kTc;
#pragma unroll 1
      for (int sl = 0; sl < slices; ++sl) {
        if (warp_ok) {
#pragma unroll 1
          for (int h = 0; h < kTc / 16; ++h) {
            const int b0 = sl * kTc + 16 * h;
            if (b0 >= p.M) break;  // warp-uniform
            float d[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(ew * 32) << 16) + kDCol + Cfg::kDStride * db + b0, d);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int b = b0 + j;
              if (b < p.M) {
                float z = d[j];
                if constexpr (byte_sum_code<CB>())
                  z = (z - static_cast<float>(1024 + byte_sum_centre<CB>()) * sh.xsum[b]) * byte_sum_scale<CB>();
                zt[(16 * h + j) * kRowBlock + row] = z;
              }
            }
          }
        }
        epi_sync();
        if (!aborted(sh)) {
          const int nb = p.M - sl * kTc < kTc ? p.M - sl * kTc : kTc;
          for (int i = et; i < nb * (kRowBlock / 4); i += 128) {
            const int bl = i / (kRowBlock / 4);
            const int q = i - bl * (kRowBlock / 4);
            const float4 v = *reinterpret_cast<const float4*>(&zt[bl * kRowBlock + 4 * q]);
            atomicAdd(reinterpret_cast<float4*>(zblk + static_cast<size_t>(sl * kTc + bl) * a.m + 4 * q), v);
          }
        }
        epi_sync();  // zt is rewritten by the next slice
      }
      if (warp_ok) tc_fence_before();
      mbar_arrive(&sh.d_empty[db]);
    }
  }

  // ---- teardown ---------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && aborted(sh) && a.status != nullptr) atomicOr(a.status, 1u);
}

// Shared memory: control block + transpose buffer + B ring + code ring.
template <int K, int NB>
inline size_t tc_smem_bytes() {
  using Cfg = TcCfg<K, NB>;
  const size_t ctrl = (sizeof(TcShared) + 1023) & ~static_cast<size_t>(1023);
  return ctrl + Cfg::kTransposeBytes + static_cast<size_t>(Cfg::kSlots) * Cfg::kBSlotBytes +
         static_cast<size_t>(Cfg::kRing) * Cfg::kChunkBytes;
}

template <int K, int CB, int NB>
exl3_status launch_tc_t(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                        cudaStream_t stream) {
  TcParams p;
  p.a = a;
  p.bimg = bimg;
  p.bsum = bsum;
  p.M = M;
  using Cfg = TcCfg<K, NB>;
  p.ct = Cfg::kWide ? 8 : (a.n % 256 == 0 ? 16 : 8);
  // At least 116 KB so that a single CTA is resident per SM (it owns all 512
  // TMEM columns; a second CTA would wait in tcgen05.alloc).
  size_t smem = tc_smem_bytes<K, NB>();
  if (smem < 116 * 1024) smem = 116 * 1024;
  if (cudaFuncSetAttribute(tc_layer_kernel<K, CB, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return EXL3_ERR_CUDA;
  const long long chunks = static_cast<long long>(a.m / kRowBlock) * (a.n / (16 * p.ct));
  if (grid > chunks) grid = static_cast<int>(chunks);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tc_layer_kernel<K, CB, NB>, p) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

// Passes of up to 128 batch rows (exl3_gemm above EXL3_MAX_BATCH rows with
// the tensor path selected): N = 128.  Skinny batches run the decode-MMA
// kernel (csrc/exl3_mv.cuh) instead.
template <int K, int CB>
exl3_status launch_tc_nb(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                         cudaStream_t stream) {
  return launch_tc_t<K, CB, kMaxNB>(a, bimg, bsum, M, grid, stream);
}

// M <= 128 batch rows; N = 128.
template <int K>
exl3_status launch_tc_dispatch(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                               cudaStream_t stream) {
  switch (a.codebook) {
    case kCb3Inst: return launch_tc_nb<K, kCb3Inst>(a, bimg, bsum, M, grid, stream);
    case kCb1Mad: return launch_tc_nb<K, kCb1Mad>(a, bimg, bsum, M, grid, stream);
    case kCbMcg: return launch_tc_nb<K, kCbMcg>(a, bimg, bsum, M, grid, stream);
    default: return launch_tc_nb<K, kCbMul1>(a, bimg, bsum, M, grid, stream);
  }
}

}  // namespace tc
}  // namespace exl3

#define EXL3_DEFINE_TC_LAUNCHER(KK)                                                                  \
  namespace exl3 {                                                                                   \
  exl3_status launch_tc_k##KK(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid, \
                              cudaStream_t stream) {                                                 \
    return tc::launch_tc_dispatch<KK>(a, bimg, bsum, M, grid, stream);                               \
  }                                                                                                  \
  }
