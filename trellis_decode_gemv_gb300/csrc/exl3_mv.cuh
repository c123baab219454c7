// Decode-MMA layer kernel for 1 <= M <= 32 batch rows (tcgen05, sm_103a):
//   y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x))))
// in one launch per call (or per group of layers) at M <= 2, and after one
// operand-image kernel above ("ExLlamaV3 & EXL3 Deep Dive" Section 2 runtime
// identity; W-hat from the bitshift-trellis codes of "Trellis Quantization"
// Parts eight and nine; 128-point blockwise transforms of Part eleven).
//
// Where the time goes at batch 1 is the decode: the integer work of the
// window, the generator and the code, per weight.  Every other step is moved
// off the decoding threads:
//  * the products go to the tensor cores: the decoded weights are written to
//    tensor memory (TMEM) as operand A of tcgen05 MMAs of 128 x N x 16 (N =
//    16 or 32 batch columns, rows past M zero), x-tilde is operand B in
//    shared memory and the fp32 accumulator D lives in TMEM;
//  * the decoders store only what the code produces:
//      byte-sum codes (1MAD, mul1): the binary16 value 1024 + S spliced by
//        dp4a, two weights paired by one byte permute; the centring,
//        -(1024 + centre) * sum(x-tilde), is one more MMA per chunk whose
//        operand A is a constant column of -(1024 + centre) in TMEM and whose
//        operand B holds the chunk's sums of x-tilde split into two binary16
//        parts (hi + lo);
//      three-instruction codes (3INST, MCG): the 32-bit mask/XOR result as
//        it is -- its two binary16 halves lo and hi are two K elements of
//        operand A, and x-tilde is duplicated in operand B, so the MMA forms
//        lo*x + hi*x without an add per weight (K doubled);
//  * the input transform is computed in the kernel by four x warps (M <= 2),
//    each taking every fourth chunk: x and the signs are loaded and rotated
//    before the warp waits for the chunk's slot, and x-tilde goes straight
//    into the operand-B slot; above M = 2 one small kernel writes the operand
//    images (and, for the byte-sum codes, their 128-column sums) once per
//    call and the x warps bulk-copy them into the slots;
//  * split-K partial sums are added into fp32 row sums in L2 (one reduction
//    per row and batch row per run), and the CTA whose arrival completes a
//    128-row block reads the row sums back, applies scale, output signs and
//    the 128-point FWHT, stores y and clears the row sums and the block's
//    counter: the output transform needs no kernel of its own.
//
// Work split: a unit is one 128-row block x one chunk of CT tile columns of
// one layer (CT = 16 for the byte-sum codes when every n is a multiple of
// 256, else 8); the units of all layers of the call, layer, block and chunk
// major, are cut into gridDim.x contiguous ranges (stream-K), one persistent
// CTA per SM.  The units of a range that share a layer and block form a run,
// accumulated in one TMEM D.
//
// Warp roles (18 warps):
//   0-7   decoders.  Warp w reaches TMEM lanes 32*(w%4) ..; thread = weight
//         row of the block (its TMEM lane), w/4 picks the half of the chunk's
//         tiles it decodes.  Per chunk: the row's code words from the
//         shared-memory ring, 16 generator outputs per tile (funnel shifts
//         give two windows each; for the three-instruction codes the second
//         window's generator output comes from the 32-bit funnel word by two
//         multiply-adds, which moves work from the ALU to the FMA pipe),
//         code, tcgen05.st of 32 or 64 columns, one arrival.
//   8     MMA issue (one lane) and TMEM allocation.
//   9     code producer: eight bulk copies (one per tile-row strip) per chunk
//         into a 2..8-deep ring.
//   10-13 x warps: operand B of each chunk (see above).
//   14-17 epilogue: D of each run out of TMEM into the row sums, the block
//         ticket and, for the completing CTA, the output transform.
// mbarriers: ring full/empty, A full/empty (3 TMEM slots), B full/empty (one
// operand-B slot per x warp), D full/empty (2 accumulators).  Every parity
// wait is on a barrier whose previous phase the waiting thread itself has
// seen complete (the decoders and the MMA lane take the chunks in order, each
// x warp owns its slot), so no wait can mistake a phase two behind for the
// one it needs.
// Every wait is bounded: on timeout the thread sets the CTA's abort flag and
// the call's status word, every role stops, the producers wait (bounded) for
// their copies in flight, the MMA lane for its MMAs, and TMEM is freed.
#pragma once

#include "exl3_tc.cuh"

namespace exl3 {
namespace mv {

using tc::bulk_g2s;
using tc::idesc_f16;
using tc::kSpinLimit;
using tc::mbar_arrive;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::mma_commit;
using tc::mma_f16_ts;
using tc::RowWords;
using tc::row_states;
using tc::smem_desc;
using tc::smem_u32;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tmem_alloc;
using tc::tmem_dealloc;
using tc::tmem_st_wait;

constexpr int kDecWarps = 8;
constexpr int kDQ = kDecWarps / 4;  // decode warps per TMEM lane quarter
constexpr int kMmaWarp = 8;
constexpr int kCodeWarp = 9;
constexpr int kXWarp0 = 10;
constexpr int kXWarps = 4;
constexpr int kEpiWarp0 = 14;
constexpr int kWarps = 18;
constexpr int kThreads = 32 * kWarps;
constexpr int kSlots = 3;        // A slots in TMEM
constexpr int kSlotCols = 128;   // TMEM columns of one A slot
constexpr int kACol = 64;        // A slots after the two D accumulators (<= 32 columns each)
constexpr int kConstCol = kACol + 3 * 128;  // 8 columns: the centring column of the byte-sum codes
constexpr int kExtK = 16;        // operand-B K elements of the centring MMA
constexpr int kTmemCols = 512;
constexpr int kMaxRing = 8;
constexpr int kRowPad = 16;      // words after each tile-row strip: lanes 16-31 read 16 banks away
constexpr int kSmemLimit = 227 * 1024;  // dynamic shared memory of one CTA
constexpr int kEpiBarrier = 2;   // named barriers (0 is __syncthreads)
constexpr int kXBarrier = 3;
constexpr int kMaxM = 32;

// Codes whose weight is an affine function of a byte sum store one binary16
// per weight (two per TMEM column); the three-instruction codes store the
// two halves of the mask/XOR word (one weight per column, K doubled).
template <int CB>
__host__ __device__ constexpr bool paired_code() {
  return byte_sum_code<CB>();
}

template <int K, int CB, int CT, int NB>
struct MvCfg {
  static constexpr bool kPaired = paired_code<CB>();
  static constexpr int kColsPerTile = kPaired ? 8 : 16;   // TMEM columns per tile row
  static constexpr int kTpt = CT / kDQ;                    // tiles per decode thread per chunk
  static constexpr int kThreadCols = kTpt * kColsPerTile;  // 64, or 32 (byte-sum codes, CT = 8)
  static constexpr int kStoreTiles = 32 / kColsPerTile;    // tiles per 32-column store
  static constexpr int kStores = kTpt / kStoreTiles;
  static constexpr int kMmas = CT * kColsPerTile / 8;      // MMAs (K = 16) per chunk
  static constexpr int kKext = 16 * kMmas;                 // operand-B K elements per chunk
  static constexpr int kBSlotBytes = (256 + kExtK) * NB * 2;  // the largest chunk + the centring block
  static constexpr int kChunkBytesB = kKext * NB * 2;
  static constexpr int kStripWords = CT * 8 * K;
  static constexpr int kRowWords = kStripWords + kRowPad;
  static constexpr int kChunkBytes = 8 * kRowWords * 4;
  // the code ring takes what the control block, the operand-B slots and the
  // output transpose buffer leave (1 KB kept spare)
  static constexpr int kRingRaw =
      (kSmemLimit - 1024 - kXWarps * kBSlotBytes - kMaxM * 128 * 4 - 1024) / kChunkBytes;
  static constexpr int kRing = kRingRaw > kMaxRing ? kMaxRing : (kRingRaw < 2 ? 2 : kRingRaw);
  static constexpr int kBlocksPerChunk = kPaired ? CT / 8 : 1;  // 128-column blocks of x per chunk
  static_assert(kTpt % kStoreTiles == 0, "store grouping");
  static_assert(kDQ * kThreadCols <= kSlotCols, "TMEM slot");
  static_assert(kACol + kSlots * kSlotCols == kConstCol && kConstCol + 8 <= kTmemCols && 2 * NB <= kACol,
                "TMEM columns");
  static_assert(kKext <= 256, "operand-B slot");
};

struct MvShared {
  uint64_t ring_full[kMaxRing];
  uint64_t ring_empty[kMaxRing];
  uint64_t a_full[kSlots];
  uint64_t a_empty[kSlots];
  uint64_t b_full[kXWarps];
  uint64_t b_empty[kXWarps];
  uint64_t d_full[2];
  uint64_t d_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t last;
  uint32_t epi_go;
};

__device__ __forceinline__ bool aborted(const MvShared& sh) {
  return *reinterpret_cast<const volatile uint32_t*>(&sh.abort) != 0u;
}
__device__ __forceinline__ void set_abort(MvShared& sh) { atomicOr(&sh.abort, 1u); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// D[tmem] += A[tmem] x B[smem desc] (accumulating; no predicate set-up per MMA).
__device__ __forceinline__ void mma_f16_ts_acc(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.eq.u32 p, 1, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc)
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, uint32_t v0) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %2, %2, %2, %2, %2, %2};" ::"r"(taddr),
               "r"(v0), "r"(0u)
               : "memory");
}

// Transaction bytes expected on an mbarrier, without an arrival.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Layer, 128-row block and chunk of unit u.
__device__ __forceinline__ void locate(const MvParams& p, int u, int& li, int& rb, int& kc) {
  li = 0;
  while (li + 1 < p.count && u >= p.l[li + 1].u_begin) ++li;
  const int lu = u - p.l[li].u_begin;
  rb = lu / p.l[li].nkb;
  kc = lu - rb * p.l[li].nkb;
}

// CTA whose stream-K range holds unit u (ranges [c*U/G, (c+1)*U/G), G <= U).
__device__ __forceinline__ int owner(long long u, long long units, long long grid) {
  return static_cast<int>(((u + 1) * grid - 1) / units);
}

// Generator outputs of the 16 steps of one tile row: the windows start at
// bits K*c (c = 0..15) of the row's words `raw` (`off` = 0 or 16: the bit
// offset of the first window in raw[0]).  When K divides 16 and K > 1 one
// 32-bit funnel word r holds the windows of steps c (top half) and c + 16/K
// (bottom half).  The second state is r - 65536 * (r >> 16); with LO_BY_IMAD
// its generator output is formed from r directly, A*r + B - (A << 16) * (r >>
// 16), two multiply-adds instead of a mask and a multiply-add (the FMA pipe
// takes the work from the ALU, for the codes whose other steps are ALU-bound).
template <int K, int CB, bool LO_BY_IMAD>
__device__ __forceinline__ void row_generate(const uint32_t (&raw)[RowWords<K>::kRaw], uint32_t off,
                                             uint32_t (&g)[16]) {
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
  constexpr uint32_t kAdd = (CB == kCbMcg || CB == kCbMul1) ? 0u : kLcgAdd;
  if constexpr (16 % K == 0 && K > 1) {
    constexpr int D = 16 / K;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      if ((c / D) % 2 == 0) {
        const uint32_t r = tc::row_bits32<K>(w, K * c);
        const uint32_t s_hi = r >> 16;
        g[c] = s_hi * kLcgMul + kAdd;
        if constexpr (LO_BY_IMAD) {
          g[c + D] = s_hi * (0u - (kLcgMul << 16)) + (r * kLcgMul + kAdd);
        } else {
          g[c + D] = (r & 0xFFFFu) * kLcgMul + kAdd;
        }
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) g[c] = (tc::row_bits32<K>(w, K * c) >> 16) * kLcgMul + kAdd;
  }
}

// One TMEM column of a byte-sum code: the binary16 values 1024 + S of two
// consecutive weights (the dp4a byte sum spliced into the mantissa of 1024),
// the first in the lower half.
template <int CB>
__device__ __forceinline__ uint32_t paired_col(uint32_t g0, uint32_t g1) {
  const uint32_t d0 = __dp4a(summed_bytes<CB>(g0), 0x01010101u, 0x6400u);
  const uint32_t d1 = __dp4a(summed_bytes<CB>(g1), 0x01010101u, 0x6400u);
  return __byte_perm(d0, d1, 0x5410);
}

template <int K, int CB, int CT, int NB, bool FUSE>
__global__ void __launch_bounds__(kThreads, 1) mv_kernel(const MvParams p) {
  using Cfg = MvCfg<K, CB, CT, NB>;
  constexpr int kRing = Cfg::kRing;
  constexpr int kTw = 8 * K;  // words per tile
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  MvShared& sh = *reinterpret_cast<MvShared*>(smem_raw);
  const size_t ctrl = (sizeof(MvShared) + 1023) & ~static_cast<size_t>(1023);
  unsigned char* bslots = smem_raw + ctrl;  // kXWarps x kBSlotBytes, 1024-aligned
  float* zt = reinterpret_cast<float*>(bslots + kXWarps * Cfg::kBSlotBytes);  // [M][128]
  uint32_t* ring = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(zt) + kMaxM * 128 * 4);

  // The next kernel on the stream may be scheduled now: it waits for this
  // grid to complete before it reads anything this grid writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const long long U = p.units;
  const long long G = gridDim.x;
  const int lo = static_cast<int>(U * blockIdx.x / G);
  const int hi = static_cast<int>(U * (blockIdx.x + 1) / G);

  // ---- set-up: barriers, TMEM; the code producer issues its first chunks first
  auto issue_chunk = [&](int seq, int u) {
    int li, rb, kc;
    locate(p, u, li, rb, kc);
    const MvLayer& L = p.l[li];
    const int slot = seq % kRing;
    if (lane == 0) mbar_arrive_expect_tx(&sh.ring_full[slot], 8u * Cfg::kStripWords * 4u);
    __syncwarp();
    if (lane < 8) {
      uint32_t* dst = ring + static_cast<size_t>(slot) * (Cfg::kChunkBytes / 4) + lane * Cfg::kRowWords;
      const uint32_t* src =
          L.codes + (static_cast<size_t>(rb * 8 + lane) * (L.n / 16) + static_cast<size_t>(kc) * CT) * kTw;
      bulk_g2s(dst, src, Cfg::kStripWords * 4u, &sh.ring_full[slot]);
    }
  };
  int pre = 0;
  if (warp == kCodeWarp) {
    if (lane == 0) {
      for (int i = 0; i < kRing; ++i) {
        mbar_init(&sh.ring_full[i], 1);
        mbar_init(&sh.ring_empty[i], kDecWarps);
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    pre = min(2, hi - lo);
    for (int s = 0; s < pre; ++s) issue_chunk(s, lo + s);
  }
  if (warp == kMmaWarp) tmem_alloc(&sh.tmem_base, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sh.a_full[i], kDecWarps);
      mbar_init(&sh.a_empty[i], 1);
    }
    for (int i = 0; i < kXWarps; ++i) {
      mbar_init(&sh.b_full[i], 1);
      mbar_init(&sh.b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.d_full[i], 1);
      mbar_init(&sh.d_empty[i], 4);
    }
    mbar_init(&sh.mma_done, 1);
    sh.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp < kDecWarps) {
    // ---- decoders ----------------------------------------------------------------
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int row = quarter * 32 + lane;  // row within the 128-row block (TMEM lane)
    const int trow = row >> 4;
    const int rr = row & 15;
    const int q0 = (rr * K) >> 1;  // first word of the row's window, and its bit offset
    const uint32_t off = static_cast<uint32_t>((rr * K) & 1) * 16u;
    const uint32_t lane_addr =
        tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kACol + half * Cfg::kThreadCols;
    if constexpr (Cfg::kPaired) {
      // The centring column: A = -(1024 + centre) at K elements 0 and 1, zero
      // elsewhere (stored once; the first a_full arrival publishes it).
      if (half == 0) {
        const uint32_t c2 =
            static_cast<uint32_t>(__half_as_ushort(__int2half_rn(-(1024 + byte_sum_centre<CB>())))) * 0x10001u;
        tmem_st8(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kConstCol, c2);
      }
    }
    // the second window of a funnel word through the FMA pipe where the
    // code's other steps load the ALU more (every code but 1MAD)
    constexpr bool kLoByImad = CB != kCb1Mad;
    int seq = 0;
    for (int u = lo; u < hi; ++u, ++seq) {
      const int rslot = seq % kRing;
      bool ok = mbar_wait(&sh.ring_full[rslot], (seq / kRing) & 1);
      if (!ok) set_abort(sh);
      if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) break;
      const uint32_t* rw = ring + static_cast<size_t>(rslot) * (Cfg::kChunkBytes / 4) + trow * Cfg::kRowWords +
                           half * Cfg::kTpt * kTw;
      const int aslot = seq % kSlots;
      const int ause = seq / kSlots;
      bool stop = false;
#pragma unroll
      for (int g = 0; g < Cfg::kStores; ++g) {
        uint32_t raw[Cfg::kStoreTiles][RowWords<K>::kRaw];
#pragma unroll
        for (int t = 0; t < Cfg::kStoreTiles; ++t) {
#pragma unroll
          for (int i = 0; i < RowWords<K>::kRaw; ++i) {
            int idx = q0 + i;
            if (idx >= kTw) idx -= kTw;
            raw[t][i] = rw[(g * Cfg::kStoreTiles + t) * kTw + idx];
          }
        }
        if (g == Cfg::kStores - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.ring_empty[rslot]);
        }
        uint32_t v[32];
#pragma unroll
        for (int t = 0; t < Cfg::kStoreTiles; ++t) {
          uint32_t gen[16];
          row_generate<K, CB, kLoByImad>(raw[t], off, gen);
          if constexpr (Cfg::kPaired) {
#pragma unroll
            for (int c = 0; c < 16; c += 2) v[t * 8 + c / 2] = paired_col<CB>(gen[c], gen[c + 1]);
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) v[t * 16 + c] = mask_xor_3inst(gen[c]);
          }
        }
        if (g == 0 && ause > 0) {
          ok = mbar_wait(&sh.a_empty[aslot], (ause - 1) & 1);
          if (!ok) set_abort(sh);
          if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) {
            stop = true;
            break;
          }
        }
        tmem_st32(lane_addr + aslot * kSlotCols + g * 32, v);
      }
      if (stop) break;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.a_full[aslot]);
    }
    tmem_st_wait();
  } else if (warp == kMmaWarp) {
    // ---- MMA issue --------------------------------------------------------------------
    constexpr uint32_t idesc = idesc_f16<NB>();
    constexpr uint32_t kLbo = (NB / 8) * 128;  // next 8 K elements
    constexpr uint32_t kSbo = 128;             // next 8 rows of N
    const uint64_t bdesc0 = smem_desc(smem_u32(bslots), kLbo, kSbo);
    int seq = 0;
    int run = 0;
    bool bad = false;
    for (int u = lo; u < hi && !bad; ++run) {
      int li, rb, kc;
      locate(p, u, li, rb, kc);
      const int end = min(hi, u + (p.l[li].nkb - kc));
      const int db = run & 1;
      const bool okd = run < 2 || mbar_wait(&sh.d_empty[db], ((run >> 1) - 1) & 1);
      if (__any_sync(0xFFFFFFFFu, !okd)) {
        set_abort(sh);
        break;
      }
      const uint32_t dt = tmem + static_cast<uint32_t>(db * NB);
      for (uint32_t acc = 0; u < end; ++u, ++seq, acc = 1) {
        const int slot = seq % kSlots;
        const int bslot = seq % kXWarps;
        const bool ok = mbar_wait(&sh.a_full[slot], (seq / kSlots) & 1) &&
                        mbar_wait(&sh.b_full[bslot], (seq / kXWarps) & 1) && !aborted(sh);
        if (__any_sync(0xFFFFFFFFu, !ok)) {
          set_abort(sh);
          bad = true;
          break;
        }
        tc_fence_after();
        const uint64_t bd = bdesc0 + ((static_cast<uint32_t>(bslot) * Cfg::kBSlotBytes) >> 4);
        const uint32_t at = tmem + kACol + slot * kSlotCols;
        if (lane == 0) {
          mma_f16_ts(dt, at, bd, idesc, acc);
#pragma unroll
          for (int j = 1; j < Cfg::kMmas; ++j) mma_f16_ts_acc(dt, at + 8 * j, bd + ((2u * j * kLbo) >> 4), idesc);
          if constexpr (Cfg::kPaired)  // the centring MMA
            mma_f16_ts_acc(dt, tmem + kConstCol, bd + ((static_cast<uint32_t>(Cfg::kKext / 8) * kLbo) >> 4), idesc);
          mma_commit(&sh.a_empty[slot]);
          mma_commit(&sh.b_empty[bslot]);
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
  } else if (warp == kCodeWarp) {
    // ---- code producer ------------------------------------------------------------------
    int seq = pre;
    for (int u = lo + pre; u < hi; ++u, ++seq) {
      const int slot = seq % kRing;
      const int use = seq / kRing;
      bool ok = true;
      if (use > 0) ok = mbar_wait(&sh.ring_empty[slot], (use - 1) & 1);
      if (!ok) set_abort(sh);
      if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) break;
      issue_chunk(seq, u);
    }
    // Every copy issued into the ring must land before the CTA exits.
    for (int i = 0; i < kRing && i < seq; ++i) {
      const int s = seq - 1 - i;
      mbar_wait(&sh.ring_full[s % kRing], (s / kRing) & 1);
    }
  } else if (warp < kXWarp0 + kXWarps) {
    // ---- operand B ----------------------------------------------------------------------
    // x warp xw produces the chunks seq = xw, xw + kXWarps, ...  The slots
    // start zeroed (rows M.., the unused K elements of the centring block);
    // afterwards only rows < M are written.
    const int xw = warp - kXWarp0;
    const int xt = tid - kXWarp0 * 32;
    {
      uint4* bz = reinterpret_cast<uint4*>(bslots);
      for (int i = xt; i < kXWarps * Cfg::kBSlotBytes / 16; i += 32 * kXWarps) bz[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    named_sync(kXBarrier, 32 * kXWarps);
    // x, the signs and the operand images may be written by the preceding
    // grid on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int M = p.M;
    unsigned char* bs = bslots + static_cast<size_t>(xw) * Cfg::kBSlotBytes;  // this warp's slot
    int last = -1;  // the last chunk this warp posted
    for (int u = lo + xw, seq = xw; u < hi; u += kXWarps, seq += kXWarps) {
      const int use = seq / kXWarps;
      int li, rb, kc;
      locate(p, u, li, rb, kc);
      const MvLayer& L = p.l[li];
      // centring sums of this chunk, per batch row (byte-sum codes)
      float csum[2] = {0.f, 0.f};
      uint2 hv[Cfg::kBlocksPerChunk * 2];
      if constexpr (FUSE) {
        // Load and rotate before waiting for the slot: the L2 latency of x
        // overlaps the MMAs still reading the slot.
        uint2 xr[Cfg::kBlocksPerChunk * 2];
        uint2 sr[Cfg::kBlocksPerChunk];
#pragma unroll
        for (int blk = 0; blk < Cfg::kBlocksPerChunk; ++blk) {
          const int col = kc * CT * 16 + blk * kRowBlock + 4 * lane;
          sr[blk] = L.s_in != nullptr ? *reinterpret_cast<const uint2*>(L.s_in + col) : make_uint2(0u, 0u);
#pragma unroll
          for (int b = 0; b < 2; ++b)
            xr[blk * 2 + b] = b < M ? *reinterpret_cast<const uint2*>(L.x + static_cast<size_t>(b) * L.n + col)
                                    : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int blk = 0; blk < Cfg::kBlocksPerChunk; ++blk) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            if (b < M) {  // warp-uniform
              const uint2 x2 = xr[blk * 2 + b];
              float v[4] = {__low2float(*reinterpret_cast<const __half2*>(&x2.x)),
                            __high2float(*reinterpret_cast<const __half2*>(&x2.x)),
                            __low2float(*reinterpret_cast<const __half2*>(&x2.y)),
                            __high2float(*reinterpret_cast<const __half2*>(&x2.y))};
              if (L.s_in != nullptr) {
                v[0] *= __low2float(*reinterpret_cast<const __half2*>(&sr[blk].x));
                v[1] *= __high2float(*reinterpret_cast<const __half2*>(&sr[blk].x));
                v[2] *= __low2float(*reinterpret_cast<const __half2*>(&sr[blk].y));
                v[3] *= __high2float(*reinterpret_cast<const __half2*>(&sr[blk].y));
                fwht128_warp(v, lane);
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
              }
              const __half2 o01 = __floats2half2_rn(v[0], v[1]);
              const __half2 o23 = __floats2half2_rn(v[2], v[3]);
              hv[blk * 2 + b].x = *reinterpret_cast<const uint32_t*>(&o01);
              hv[blk * 2 + b].y = *reinterpret_cast<const uint32_t*>(&o23);
              if constexpr (Cfg::kPaired)
                csum[b] += (__low2float(o01) + __high2float(o01)) + (__low2float(o23) + __high2float(o23));
            }
          }
        }
      } else if constexpr (Cfg::kPaired) {
        // the chunk's sums of the binary16 operand values, from the image kernel
        const int nblk = L.n / kRowBlock;
#pragma unroll
        for (int blk = 0; blk < Cfg::kBlocksPerChunk; ++blk) {
          const int b = lane;
          if (b < M) csum[0] += __ldcg(L.bsum + static_cast<size_t>(b) * nblk + kc * Cfg::kBlocksPerChunk + blk);
        }
      }
      // wait until the MMAs of the slot's previous chunk are done with it
      bool ok = true;
      if (use > 0) ok = mbar_wait(&sh.b_empty[xw], (use - 1) & 1);
      if (!ok) set_abort(sh);
      if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) break;
      if constexpr (!FUSE) {
        if (lane == 0 && p.debug_stall == 0) {
          mbar_expect_tx(&sh.b_full[xw], Cfg::kChunkBytesB);
          bulk_g2s(bs, L.bimg + static_cast<size_t>(kc) * Cfg::kKext * NB, Cfg::kChunkBytesB, &sh.b_full[xw]);
        }
      } else {
#pragma unroll
        for (int blk = 0; blk < Cfg::kBlocksPerChunk; ++blk) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            if (b < M) {
              if constexpr (Cfg::kPaired) {
                // K elements k = blk*128 + 4*lane .. +3: half a 16-byte core row
                const int k = blk * kRowBlock + 4 * lane;
                *reinterpret_cast<uint2*>(bs + ((k >> 3) * (NB / 8) + (b >> 3)) * 128 + (b & 7) * 16 + (k & 7) * 2) =
                    hv[blk * 2 + b];
              } else {
                // K elements 8*lane .. 8*lane+7: columns 4*lane .. 4*lane+3, each twice
                const uint2 h = hv[blk * 2 + b];
                uint4 o;
                o.x = (h.x & 0xFFFFu) * 0x10001u;
                o.y = (h.x >> 16) * 0x10001u;
                o.z = (h.y & 0xFFFFu) * 0x10001u;
                o.w = (h.y >> 16) * 0x10001u;
                *reinterpret_cast<uint4*>(bs + (lane * (NB / 8) + (b >> 3)) * 128 + (b & 7) * 16) = o;
              }
            }
          }
        }
      }
      if constexpr (Cfg::kPaired) {
        // Sum of the chunk's operand values per batch row, as hi + lo in
        // binary16 at K elements kKext and kKext + 1 of the centring block.
        float sums[2] = {csum[0], csum[1]};
        if constexpr (FUSE) {
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) sums[b] += __shfl_xor_sync(0xFFFFFFFFu, sums[b], d);
        }
        constexpr int ke = Cfg::kKext;
        if constexpr (FUSE) {
          if (lane < M) {
            const float sv = lane == 0 ? sums[0] : sums[1];
            const __half h = __float2half_rn(sv);
            const __half l = __float2half_rn(sv - __half2float(h));
            *reinterpret_cast<__half2*>(bs + ((ke >> 3) * (NB / 8) + (lane >> 3)) * 128 + (lane & 7) * 16) =
                __halves2half2(h, l);
          }
        } else {
          if (lane < M) {
            const __half h = __float2half_rn(sums[0]);
            const __half l = __float2half_rn(sums[0] - __half2float(h));
            *reinterpret_cast<__half2*>(bs + ((ke >> 3) * (NB / 8) + (lane >> 3)) * 128 + (lane & 7) * 16) =
                __halves2half2(h, l);
          }
        }
      }
      // generic-proxy stores, read by the tensor core (async proxy)
      fence_proxy_async_smem();
      __syncwarp();
      // With the failure-detection test hook set operand B is never posted,
      // so the MMA lane's bounded wait runs out.
      if (lane == 0 && p.debug_stall == 0) mbar_arrive(&sh.b_full[xw]);
      last = seq;
    }
    if constexpr (!FUSE) {
      // The bulk copy of the last chunk posted must land before the CTA
      // exits (every earlier one was consumed before this warp waited for
      // its slot again); only this warp moves its slot's b_full phases.
      if (lane == 0 && p.debug_stall == 0 && last >= 0) mbar_wait(&sh.b_full[xw], (last / kXWarps) & 1);
    }
  } else {
    // ---- epilogue ---------------------------------------------------------------------
    // The row sums, counters and y may be in use by the preceding grid.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int ew = warp & 3;  // TMEM lane quarter
    const int et = tid - kEpiWarp0 * 32;
    const int row = ew * 32 + lane;
    const int M = p.M;
    const float factor = x_factor<CB>();
    int run = 0;
    for (int u = lo; u < hi; ++run) {
      int li, rb, kc;
      locate(p, u, li, rb, kc);
      const MvLayer& L = p.l[li];
      const int u_first = L.u_begin + rb * L.nkb;
      const int need = owner(u_first + L.nkb - 1, U, G) - owner(u_first, U, G) + 1;
      u = min(hi, u + (L.nkb - kc));
      const int db = run & 1;
      const bool ok = !aborted(sh) && mbar_wait(&sh.d_full[db], (run >> 1) & 1);
      if (!ok) set_abort(sh);
      // The four epilogue warps share named barriers: they stop together, on
      // one decision taken after all of them have waited.
      named_sync(kEpiBarrier, 128);
      if (et == 0) sh.epi_go = aborted(sh) ? 0u : 1u;
      named_sync(kEpiBarrier, 128);
      if (sh.epi_go == 0u) break;
      tc_fence_after();
      float d[NB];
      {
        float d16[16];
        tc::tmem_ld16(tmem + (static_cast<uint32_t>(ew * 32) << 16) + db * NB, d16);
#pragma unroll
        for (int j = 0; j < 16; ++j) d[j] = d16[j];
        if constexpr (NB > 16) {
          tc::tmem_ld16(tmem + (static_cast<uint32_t>(ew * 32) << 16) + db * NB + 16, d16);
#pragma unroll
          for (int j = 0; j < 16; ++j) d[16 + j] = d16[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.d_empty[db]);
      float* zrow = L.zacc + static_cast<size_t>(rb) * kRowBlock + row;
#pragma unroll
      for (int b = 0; b < NB; ++b)
        if (b < M) atomicAdd(zrow + static_cast<size_t>(b) * L.m, d[b] * factor);
      // The block's ticket: this run's sums are visible at device scope
      // before the count moves.
      fence_acq_rel_gpu();
      named_sync(kEpiBarrier, 128);
      if (et == 0) {
        const uint32_t old = atomicAdd(L.cnt + rb, 1u);
        sh.last = (old + 1u == static_cast<uint32_t>(need)) ? 1u : 0u;
      }
      named_sync(kEpiBarrier, 128);
      if (sh.last != 0u) {
        // Every partial sum of the block has arrived: finish it.
        fence_acq_rel_gpu();
        const float sc = __half2float(L.scales[rb * kRowBlock + row]);
        const float so = L.s_out != nullptr ? __half2float(L.s_out[rb * kRowBlock + row]) : 1.f;
        for (int b = 0; b < M; ++b) {
          float* zp = zrow + static_cast<size_t>(b) * L.m;
          zt[b * kRowBlock + row] = __ldcg(zp) * sc * so;
          __stcg(zp, 0.f);
        }
        if (et == 0) L.cnt[rb] = 0u;
        named_sync(kEpiBarrier, 128);
        for (int b = ew; b < M; b += 4) {
          float v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = zt[b * kRowBlock + 4 * lane + j];
          if (L.s_out != nullptr) {
            fwht128_warp(v, lane);
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
          }
          const __half2 o01 = __floats2half2_rn(v[0], v[1]);
          const __half2 o23 = __floats2half2_rn(v[2], v[3]);
          uint2 o;
          o.x = *reinterpret_cast<const uint32_t*>(&o01);
          o.y = *reinterpret_cast<const uint32_t*>(&o23);
          *reinterpret_cast<uint2*>(L.y + static_cast<size_t>(b) * L.m + rb * kRowBlock + 4 * lane) = o;
        }
        named_sync(kEpiBarrier, 128);  // zt and sh.last are rewritten by the next run
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
  if (tid == 0 && aborted(sh) && p.status != nullptr) atomicOr(p.status, 1u);
}

template <int K, int CB, int CT, int NB>
inline size_t mv_smem_bytes() {
  using Cfg = MvCfg<K, CB, CT, NB>;
  const size_t ctrl = (sizeof(MvShared) + 1023) & ~static_cast<size_t>(1023);
  return ctrl + static_cast<size_t>(kXWarps) * Cfg::kBSlotBytes + static_cast<size_t>(kMaxM) * 128 * 4 +
         static_cast<size_t>(Cfg::kRing) * Cfg::kChunkBytes;
}

template <int K, int CB, int CT, int NB, bool FUSE>
exl3_status launch_mv_t(const MvParams& p, int grid, cudaStream_t stream) {
  size_t smem = mv_smem_bytes<K, CB, CT, NB>();
  // At least 116 KB so that a single CTA is resident per SM (it owns all 512
  // TMEM columns; a second CTA would wait in tcgen05.alloc).
  if (smem < 116 * 1024) smem = 116 * 1024;
  if (cudaFuncSetAttribute(mv_kernel<K, CB, CT, NB, FUSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return EXL3_ERR_CUDA;
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
  if (cudaLaunchKernelEx(&cfg, mv_kernel<K, CB, CT, NB, FUSE>, p) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

// Tiles per chunk: 16 for the byte-sum codes when ct16 (every n a multiple
// of 256), else 8; N = 16 up to 16 batch rows, else 32; the x warps compute
// x-tilde for M <= 2.
template <int K, int CB>
exl3_status launch_mv_cb(const MvParams& p, int grid, bool ct16, cudaStream_t stream) {
  const bool fuse = p.M <= 2;
  if constexpr (paired_code<CB>()) {
    if (ct16) {
      if (fuse) return launch_mv_t<K, CB, 16, 16, true>(p, grid, stream);
      if (p.M <= 16) return launch_mv_t<K, CB, 16, 16, false>(p, grid, stream);
      return launch_mv_t<K, CB, 16, 32, false>(p, grid, stream);
    }
  }
  if (fuse) return launch_mv_t<K, CB, 8, 16, true>(p, grid, stream);
  if (p.M <= 16) return launch_mv_t<K, CB, 8, 16, false>(p, grid, stream);
  return launch_mv_t<K, CB, 8, 32, false>(p, grid, stream);
}

template <int K>
exl3_status launch_mv_dispatch(const MvParams& p, int codebook, int grid, bool ct16, cudaStream_t stream) {
  switch (codebook) {
    case kCb3Inst: return launch_mv_cb<K, kCb3Inst>(p, grid, ct16, stream);
    case kCb1Mad: return launch_mv_cb<K, kCb1Mad>(p, grid, ct16, stream);
    case kCbMcg: return launch_mv_cb<K, kCbMcg>(p, grid, ct16, stream);
    default: return launch_mv_cb<K, kCbMul1>(p, grid, ct16, stream);
  }
}

}  // namespace mv
}  // namespace exl3

#define EXL3_DEFINE_MV_LAUNCHER(KK)                                                                  \
  namespace exl3 {                                                                                   \
  exl3_status launch_mv_k##KK(const MvParams& p, int codebook, int grid, bool ct16,                  \
                              cudaStream_t stream) {                                                 \
    return mv::launch_mv_dispatch<KK>(p, codebook, grid, ct16, stream);                              \
  }                                                                                                  \
  }
