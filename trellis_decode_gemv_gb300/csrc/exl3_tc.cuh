// Fused layer kernel, tensor-core path (tcgen05, sm_103a):
//   y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x))))   for 1 <= M <= 32.
//
// The decoded 16x16 tiles feed tcgen05 MMAs directly from tensor memory:
//
//  * Operand A (128 weight rows x K) lives in TMEM.  Each decode thread owns one
//    weight row of a 128-row block (TMEM lane = row) and, per pipeline stage,
//    decodes 32 consecutive weights of that row (one row of two adjacent 16x16
//    tiles), writing two binary16 weights per 32-bit TMEM column with
//    tcgen05.st (the lower half holds the even K element).  3INST weights are
//    the binary16 sums of the two halves of the mask/XOR step ("Trellis
//    Quantization" Part nine), formed for two columns at once by two byte
//    permutes and one packed add -- exactly the defined binary16 weights; 1MAD
//    weights are stored as the half 1024 + S (the dp4a byte sum spliced into
//    the mantissa of 1024, the int-to-half trick of Part three), paired by one
//    byte permute.
//  * Operand B (K x N, N = batch padded to 16 or 32) is the rotated x slice in
//    shared memory, binary16, in the canonical K-major no-swizzle layout
//    (8x16-byte core matrices).
//  * D (128 x N fp32) accumulates in TMEM.  For 1MAD, D = sum (1024 + S) x, so
//    z = C (D - 1534 sum x) with C = 1/sqrt(21845).
//
// Persistent kernel, one CTA per SM.  Work item = one 128-row output block x
// one slice of the input dimension (a multiple of 128 columns); CTA b takes
// items b, b + gridDim.x, ...  Warp roles:
//   warps 0-15  decode: four warpgroups; warpgroup g decodes tile columns
//               2g, 2g+1 of every 8-tile-column chunk (a warp only reaches its
//               own 32-lane quarter of TMEM, so the four warps of a warpgroup
//               cover the 128 rows);
//   warps 16-19 epilogue: lay out the x slice (B) of the next item (the
//               host rotates x once per call with the standalone transform
//               kernel; these warps wait for it) and finish the
//               previous item (tcgen05.ld of D, split-K partial sums + an atomic
//               ticket per row block, and for the last slice the scale, output
//               signs, FWHT and binary16 store);
//   warp 20     MMA issue (one lane) and TMEM allocation;
//   warp 21     producer: 1-D bulk copies (cp.async.bulk) of each chunk's eight
//               tile-row strips of packed codes (one lane per strip) into a
//               4- or 8-deep shared-memory ring.
// mbarriers: ring full/empty (codes), A full/empty (8 TMEM slots), B full (2
// buffers), D full/empty (2 TMEM accumulators).  Every wait is bounded: on
// timeout the thread sets the CTA's abort flag and the workspace status word,
// every role stops, the producer waits (bounded) for its copies in flight, the
// MMA lane for its MMAs, TMEM is freed and the CTA exits.
#pragma once

#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {
namespace tc {

constexpr int kDecodeWarps = 16;
constexpr int kEpiWarp0 = 16;
constexpr int kMmaWarp = 20;
constexpr int kTmaWarp = 21;
constexpr int kThreads = 22 * 32;
constexpr int kChunkTiles = 8;          // tile columns per code chunk (128 columns)
// Code chunks in flight: 8 for K <= 4, 4 above (shared-memory budget).
template <int K>
__host__ __device__ constexpr int ring_depth() {
  return K <= 4 ? 8 : 4;
}
constexpr int kMaxRing = 8;
constexpr int kSlots = 8;               // A stages in TMEM
constexpr int kStageWeights = 32;       // weights per row per stage (two tiles)
constexpr int kStageCols = 16;          // TMEM columns per stage (two weights each)
constexpr int kTmemCols = 512;
constexpr int kDCol = 0;                // D buffers at columns 0 and 32
constexpr int kACol = 64;               // A slots at 64 + 16 * slot
constexpr int kRowPadWords = 16;        // keeps tile-row strips 64 B apart from a bank multiple
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
  const uint32_t x0 = lcg(s0);
  const uint32_t x1 = lcg(s1);
  if constexpr (CB == kCb3Inst) {
    const uint32_t h0 = mask_xor_3inst(x0);
    const uint32_t h1 = mask_xor_3inst(x1);
    const uint32_t lo = __byte_perm(h0, h1, 0x5410);  // (lo half of w0, lo half of w1)
    const uint32_t hi = __byte_perm(h0, h1, 0x7632);  // (hi half of w0, hi half of w1)
    const __half2 w = __hadd2(*reinterpret_cast<const __half2*>(&lo), *reinterpret_cast<const __half2*>(&hi));
    return *reinterpret_cast<const uint32_t*>(&w);
  } else {
    const uint32_t d0 = __dp4a(x0, 0x01010101u, 0x6400u);  // binary16 bits of 1024 + S
    const uint32_t d1 = __dp4a(x1, 0x01010101u, 0x6400u);
    return __byte_perm(d0, d1, 0x5410);
  }
}

struct TcParams {
  LayerArgs a;
  int M;
  int ns;          // slice width (columns), multiple of 128
  int nslices;     // n / ns
  int items;       // (m / 128) * nslices
};

struct TcShared {
  uint64_t ring_full[kMaxRing];
  uint64_t ring_empty[kMaxRing];
  uint64_t a_full[kSlots];
  uint64_t a_empty[kSlots];
  uint64_t b_full[2];
  uint64_t d_full[2];
  uint64_t d_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t ticket;
  uint32_t epi_go;
  float xsum[2][32];
  float zs[32 * 128];
};

template <int K>
__host__ __device__ constexpr int chunk_row_words() {
  return kChunkTiles * 8 * K + kRowPadWords;
}
template <int K>
__host__ __device__ constexpr int chunk_bytes() {
  return 8 * chunk_row_words<K>() * 4;
}

__device__ __forceinline__ bool aborted(const TcShared& sh) {
  return *reinterpret_cast<const volatile uint32_t*>(&sh.abort) != 0u;
}

__device__ __forceinline__ void set_abort(TcShared& sh) { atomicOr(&sh.abort, 1u); }

template <int K, int CB, int NB>
__global__ void __launch_bounds__(kThreads, 1) tc_layer_kernel(TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  TcShared& sh = *reinterpret_cast<TcShared*>(smem_raw);
  const size_t ctrl = (sizeof(TcShared) + 1023) & ~static_cast<size_t>(1023);
  uint32_t* ring = reinterpret_cast<uint32_t*>(smem_raw + ctrl);
  constexpr int kRing = ring_depth<K>();
  unsigned char* bbuf = smem_raw + ctrl + static_cast<size_t>(kRing) * chunk_bytes<K>();
  const size_t bbytes = static_cast<size_t>(NB) * p.ns * sizeof(__half);

  const LayerArgs& a = p.a;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int tiles_per_row = a.n / 16;
  const int nst_item = p.ns / kStageWeights;
  const int nchunk_item = p.ns / (kChunkTiles * 16);
  // items of this CTA: blockIdx.x + i * gridDim.x
  const int my_items = p.items > static_cast<int>(blockIdx.x)
                           ? (p.items - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                           : 0;

  // ---- set-up ---------------------------------------------------------------
  if (warp == kMmaWarp) tmem_alloc(&sh.tmem_base, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&sh.ring_full[i], 1);
      mbar_init(&sh.ring_empty[i], kDecodeWarps);  // one elected arrival per decode warp
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sh.a_full[i], 4);  // one elected arrival per warp of the warpgroup
      mbar_init(&sh.a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.b_full[i], 128);
      mbar_init(&sh.d_full[i], 1);
      mbar_init(&sh.d_empty[i], 128);
    }
    mbar_init(&sh.mma_done, 1);
    sh.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // B rows n >= M stay zero for the whole kernel.
  for (size_t i = static_cast<size_t>(tid) * 16; i < 2 * bbytes; i += static_cast<size_t>(kThreads) * 16)
    *reinterpret_cast<uint4*>(bbuf + i) = make_uint4(0, 0, 0, 0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kTmaWarp) {
    // ---- producer: code chunks into the ring ----------------------------------
    // Lanes 0-7 each copy one tile-row strip of a chunk; lane 0 posts the
    // expected byte count first.
    int seq = 0;
    bool stop = false;
    for (int li = 0; li < my_items && !stop; ++li) {
      const int item = static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x);
      const int rb = item / p.nslices;
      const int sl = item - rb * p.nslices;
      for (int ch = 0; ch < nchunk_item; ++ch, ++seq) {
        const int slot = seq % kRing;
        const int use = seq / kRing;
        bool ok = true;
        if (use > 0) ok = mbar_wait(&sh.ring_empty[slot], (use - 1) & 1);
        if (!ok) set_abort(sh);
        if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) {
          stop = true;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&sh.ring_full[slot], 8u * kChunkTiles * 32u * K);
        __syncwarp();
        if (lane < 8) {
          const int J0 = (sl * p.ns) / 16 + ch * kChunkTiles;
          uint32_t* dst = ring + static_cast<size_t>(slot) * (chunk_bytes<K>() / 4);
          const uint32_t* src =
              a.codes + (static_cast<size_t>(rb * 8 + lane) * tiles_per_row + J0) * (8 * K);
          bulk_g2s(dst + lane * chunk_row_words<K>(), src, kChunkTiles * 32u * K, &sh.ring_full[slot]);
        }
      }
    }
    // Wait (bounded) for every copy issued into the ring to land before exit.
    for (int i = 0; i < kRing && i < seq; ++i) {
      const int s = seq - 1 - i;
      mbar_wait(&sh.ring_full[s % kRing], (s / kRing) & 1);
    }
  } else if (warp < kDecodeWarps) {
    // ---- decode producers of operand A -------------------------------------------
    const int g = warp >> 2;              // warpgroup: stage g of every chunk
    const int quarter = warp & 3;         // TMEM lanes 32 * quarter ..
    const int row = quarter * 32 + lane;  // row within the 128-row block
    const int trow = row >> 4;            // tile row within the block
    const int rr = row & 15;
    const int q0 = (rr * K) >> 1;
    const uint32_t off = static_cast<uint32_t>((rr * K) & 1) * 16u;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int seq = 0;
    bool stop = false;
    for (int li = 0; li < my_items && !stop; ++li) {
      for (int ch = 0; ch < nchunk_item; ++ch, ++seq) {
        const int slot = seq % kRing;
        bool ok = mbar_wait(&sh.ring_full[slot], (seq / kRing) & 1);
        if (!ok) set_abort(sh);
        if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) {
          stop = true;
          break;
        }
        const uint32_t* rw = ring + static_cast<size_t>(slot) * (chunk_bytes<K>() / 4) +
                             trow * chunk_row_words<K>() + (2 * g) * (8 * K);
        uint32_t raw0[RowWords<K>::kRaw], raw1[RowWords<K>::kRaw];
#pragma unroll
        for (int i = 0; i < RowWords<K>::kRaw; ++i) {
          int idx = q0 + i;
          if (idx >= 8 * K) idx -= 8 * K;
          raw0[i] = rw[idx];
          raw1[i] = rw[8 * K + idx];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.ring_empty[slot]);
        uint32_t st0[16], st1[16];
        row_states<K>(raw0, off, st0);
        row_states<K>(raw1, off, st1);
        uint32_t v[16];
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          v[c / 2] = pack_two<CB>(st0[c], st0[c + 1]);
          v[8 + c / 2] = pack_two<CB>(st1[c], st1[c + 1]);
        }
        const int gs = 4 * seq + g;  // global stage index of this CTA
        const int aslot = gs % kSlots;
        const int use = gs / kSlots;
        ok = true;
        if (use > 0) ok = mbar_wait(&sh.a_empty[aslot], (use - 1) & 1);
        if (!ok) set_abort(sh);
        if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) {
          stop = true;
          break;
        }
        tmem_st16(lane_addr + kACol + aslot * kStageCols, v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.a_full[aslot]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issue ------------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16<NB>();
      constexpr uint32_t kLbo = (NB / 8) * 128;  // next 8 K-elements
      constexpr uint32_t kSbo = 128;             // next 8 rows of N
      int gs = 0;
      for (int li = 0; li < my_items && !aborted(sh); ++li) {
        const int db = li & 1;
        if (!mbar_wait(&sh.b_full[db], (li >> 1) & 1)) {
          set_abort(sh);
          break;
        }
        if (li >= 2 && !mbar_wait(&sh.d_empty[db], ((li >> 1) - 1) & 1)) {
          set_abort(sh);
          break;
        }
        tc_fence_after();
        const uint32_t bbase = smem_u32(bbuf + db * bbytes);
        bool bad = false;
        for (int s = 0; s < nst_item; ++s, ++gs) {
          const int aslot = gs % kSlots;
          if (!mbar_wait(&sh.a_full[aslot], (gs / kSlots) & 1) || aborted(sh)) {
            set_abort(sh);
            bad = true;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t kk = static_cast<uint32_t>(s) * kStageWeights + 16u * j;  // K offset
            const uint64_t bd = smem_desc(bbase + (kk / 8) * kLbo, kLbo, kSbo);
            mma_f16_ts(tmem + kDCol + 32 * db, tmem + kACol + aslot * kStageCols + 8 * j, bd, idesc,
                       (s > 0 || j > 0) ? 1u : 0u);
          }
          mma_commit(&sh.a_empty[aslot]);
        }
        if (bad) break;
        mma_commit(&sh.d_full[db]);
      }
      mma_commit(&sh.mma_done);
      mbar_wait(&sh.mma_done, 0);
    }
  } else {
    // ---- epilogue warps: B of the next item, finish the previous one ----------------
    const int ew = warp - kEpiWarp0;  // 0..3 = TMEM lane quarter
    const int et = tid - kEpiWarp0 * 32;  // 0..127
    const int nkb = p.ns / kRowBlock;
    // x may be written by the preceding kernel on the stream (the rotation).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int li = 0; li <= my_items; ++li) {
      // Uniform go/stop decision for the four epilogue warps: they share named
      // barriers, so they must leave together.
      if (et == 0) sh.epi_go = aborted(sh) ? 0u : 1u;
      epi_sync();
      if (sh.epi_go == 0u) break;
      if (li < my_items) {
        // B[li & 1] for item li (free: the MMAs of item li-2 finished before the
        // epilogue of item li-2 ran in the previous iteration).
        const int db = li & 1;
        const int item = static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x);
        const int sl = item % p.nslices;
        const int c0 = sl * p.ns;
        unsigned char* bsm = bbuf + db * bbytes;
        if (et < 32) sh.xsum[db][et] = 0.f;
        epi_sync();
        for (int job = ew; job < p.M * nkb; job += 4) {
          const int n = job / nkb;
          const int kb = job - n * nkb;
          const int col = c0 + kb * kRowBlock + 4 * lane;
          float v[4];
          {
            const uint2 xr = *reinterpret_cast<const uint2*>(a.x + static_cast<size_t>(n) * a.n + col);
            const __half2 x01 = *reinterpret_cast<const __half2*>(&xr.x);
            const __half2 x23 = *reinterpret_cast<const __half2*>(&xr.y);
            v[0] = __low2float(x01);
            v[1] = __high2float(x01);
            v[2] = __low2float(x23);
            v[3] = __high2float(x23);
          }
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
          __half h[4];
          float hs = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            h[j] = __float2half_rn(v[j]);
            hs += __half2float(h[j]);
          }
          // element (n, k) at ((k/8) * (NB/8) + n/8) * 128 + (n%8) * 16 + (k%8) * 2;
          // these four values are k = kb*128 + 4*lane .. +3.
          const int kc = kb * 16 + lane / 2;
          const uint32_t o = (static_cast<uint32_t>(kc) * (NB / 8) + n / 8) * 128u + (n % 8) * 16u +
                             (lane % 2) * 8u;
          uint2 pk;
          pk.x = static_cast<uint32_t>(__half_as_ushort(h[0])) |
                 (static_cast<uint32_t>(__half_as_ushort(h[1])) << 16);
          pk.y = static_cast<uint32_t>(__half_as_ushort(h[2])) |
                 (static_cast<uint32_t>(__half_as_ushort(h[3])) << 16);
          *reinterpret_cast<uint2*>(bsm + o) = pk;
          if (CB == kCb1Mad) {
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) hs += __shfl_xor_sync(0xFFFFFFFFu, hs, d);
            if (lane == 0) atomicAdd(&sh.xsum[db][n], hs);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        epi_sync();
        mbar_arrive(&sh.b_full[db]);
      }
      if (li >= 1) {
        // finish item li-1
        const int pi = li - 1;
        const int db = pi & 1;
        const int item = static_cast<int>(blockIdx.x) + pi * static_cast<int>(gridDim.x);
        const int rb = item / p.nslices;
        const int sl = item - rb * p.nslices;
        bool ok = !aborted(sh) && mbar_wait(&sh.d_full[db], (pi >> 1) & 1);
        if (!ok) set_abort(sh);
        // tcgen05.ld is a whole-warp instruction: skip it warp-uniformly.
        if (!__any_sync(0xFFFFFFFFu, !ok)) {
          tc_fence_after();
          const int row = ew * 32 + lane;
          float d[16];
          tmem_ld16(tmem + (static_cast<uint32_t>(ew * 32) << 16) + kDCol + 32 * db, d);
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            if (n < p.M) {
              float z = d[n];
              if (CB == kCb1Mad) z = (z - 1534.0f * sh.xsum[db][n]) * kOneMadScale;
              sh.zs[n * kRowBlock + row] = z;
            }
          }
          if constexpr (NB == 32) {
            tmem_ld16(tmem + (static_cast<uint32_t>(ew * 32) << 16) + kDCol + 32 * db + 16, d);
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              if (16 + n < p.M) {
                float z = d[n];
                if (CB == kCb1Mad) z = (z - 1534.0f * sh.xsum[db][16 + n]) * kOneMadScale;
                sh.zs[(16 + n) * kRowBlock + row] = z;
              }
            }
          }
          tc_fence_before();
        }
        mbar_arrive(&sh.d_empty[db]);
        epi_sync();
        bool last = true;
        if (p.nslices > 1) {
          float* part = a.partials + static_cast<size_t>(sl) * p.M * a.m;
          for (int i = et; i < p.M * kRowBlock; i += 128) {
            const int b = i / kRowBlock;
            const int r = i - b * kRowBlock;
            part[static_cast<size_t>(b) * a.m + rb * kRowBlock + r] = sh.zs[i];
          }
          __threadfence();
          epi_sync();
          if (et == 0) sh.ticket = atomicAdd(a.counters + rb, 1u);
          epi_sync();
          last = sh.ticket == static_cast<uint32_t>(p.nslices - 1);
          if (last) {
            __threadfence();
            for (int i = et; i < p.M * kRowBlock; i += 128) {
              const int b = i / kRowBlock;
              const int r = i - b * kRowBlock;
              float acc = 0.f;
              for (int sp = 0; sp < p.nslices; ++sp)
                acc += __ldcg(a.partials + (static_cast<size_t>(sp) * p.M + b) * a.m + rb * kRowBlock + r);
              sh.zs[i] = acc;
            }
            if (et == 0) a.counters[rb] = 0u;
            epi_sync();
          }
        }
        if (last) {
          for (int b = ew; b < p.M; b += 4) {
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
        epi_sync();  // zs is reused by the next item
      }
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

// Shared memory: control block + code ring + two B buffers (NB x ns halves).
template <int K>
inline size_t tc_smem_bytes(int nb, int ns) {
  const size_t ctrl = (sizeof(TcShared) + 1023) & ~static_cast<size_t>(1023);
  return ctrl + static_cast<size_t>(ring_depth<K>()) * chunk_bytes<K>() +
         2 * static_cast<size_t>(nb) * ns * sizeof(__half);
}

template <int K, int CB, int NB>
exl3_status launch_tc_t(const LayerArgs& a, int M, int ns, int grid, cudaStream_t stream) {
  TcParams p;
  p.a = a;
  p.M = M;
  p.ns = ns;
  p.nslices = a.n / ns;
  p.items = (a.m / kRowBlock) * p.nslices;
  // At least 116 KB so that a single CTA is resident per SM (it owns all 512
  // TMEM columns; a second CTA would wait in tcgen05.alloc).
  size_t smem = tc_smem_bytes<K>(NB, ns);
  if (smem < 116 * 1024) smem = 116 * 1024;
  if (cudaFuncSetAttribute(tc_layer_kernel<K, CB, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return EXL3_ERR_CUDA;
  if (grid > p.items) grid = p.items;
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

template <int K>
exl3_status launch_tc_dispatch(const LayerArgs& a, int M, int ns, int grid, cudaStream_t stream) {
  if (a.codebook == kCb3Inst)
    return M <= 16 ? launch_tc_t<K, kCb3Inst, 16>(a, M, ns, grid, stream)
                   : launch_tc_t<K, kCb3Inst, 32>(a, M, ns, grid, stream);
  return M <= 16 ? launch_tc_t<K, kCb1Mad, 16>(a, M, ns, grid, stream)
                 : launch_tc_t<K, kCb1Mad, 32>(a, M, ns, grid, stream);
}

}  // namespace tc
}  // namespace exl3

#define EXL3_DEFINE_TC_LAUNCHER(KK)                                                           \
  namespace exl3 {                                                                            \
  exl3_status launch_tc_k##KK(const LayerArgs& a, int M, int ns, int grid, cudaStream_t stream) { \
    return tc::launch_tc_dispatch<KK>(a, M, ns, grid, stream);                                \
  }                                                                                           \
  }
