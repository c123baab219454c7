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
//  * the decoders store one binary16 value per weight, two per TMEM column:
//      byte-sum codes (1MAD, mul1): 1024 + S, the dp4a byte sum spliced into
//        the mantissa of 1024; the centring, -(1024 + centre) * sum(x-tilde),
//        is one more MMA per chunk whose operand A is a constant column of
//        -(1024 + centre) in TMEM and whose operand B holds the chunk's sums
//        of x-tilde split into two binary16 parts (hi + lo);
//      three-instruction codes (3INST, MCG): the defined weight, the binary16
//        sum lo + hi of the two halves of the mask/XOR word (one packed add on
//        the word's halves per weight, one byte permute per pair).  Storing lo
//        and hi as two K elements would save those instructions but double
//        the MMAs, and at 128 x N x 16 the tensor core takes about 50 cycles
//        per MMA whatever N <= 64 is;
//  * the input transform is computed in the kernel (M <= 2): x and the signs
//    are loaded and rotated before the slot is free, and x-tilde goes straight
//    into the operand-B slot; above M = 2 one small kernel writes the operand
//    images (and, for the byte-sum codes, their 128-column sums) once per
//    call and they are bulk-copied into the slots;
//  * split-K partial sums are added into fp32 row sums in L2 (one reduction
//    per row and batch row per run), and the CTA whose arrival completes a
//    128-row block reads the row sums back, applies scale, output signs and
//    the 128-point FWHT, stores y and clears the row sums and the block's
//    counter: the output transform needs no kernel of its own.
//
// MMA issue.  A tcgen05.mma is issued by one thread, and that thread's warp
// competes for its scheduler with the decoders of the same SM sub-partition
// (a TMEM lane quarter belongs to one sub-partition, so every sub-partition
// decodes): measured, a lone issuer beside busy warps of its own
// sub-partition stalls for hundreds of cycles per MMA, against about 50 for
// the tensor core.  So six issuers, spread over the sub-partitions, share the
// MMAs: issuer i takes the chunks seq = i (mod 6) and owns A slot i and B
// slot i (six slots also keep each decoder team two chunks ahead of the MMAs
// it waits for).
// D is zeroed by the epilogue when it takes a run's sums out, so every MMA
// accumulates and the order in which the issuers' MMAs reach the tensor core
// does not matter.
//
// Work split: a unit is one 128-row block x one chunk of 8 tile columns (128
// input columns) of one layer; the units of all layers of the call, layer,
// block and chunk major, are cut into gridDim.x contiguous ranges (stream-K),
// one persistent CTA per SM.  The units of a range that share a layer and
// block form a run, accumulated in one TMEM D.
//
// Warp roles (22 warps):
//   0-11  decoders, three teams of four: warp w reaches TMEM lanes 32*(w%4) ..
//         (thread = weight row of the block), team w/4 takes the chunks seq
//         = w/4 (mod 3).  The team's lead lane loads each of its chunks' codes
//         with one 2-D tensor copy (the 8 tile-row strips of the chunk, the
//         codes viewed as (m/16) rows of (n/16)*8K words) into the shared-
//         memory ring.  Per chunk a thread: the row's code words of 8 tiles,
//         16 generator outputs per tile (funnel shifts give two windows each;
//         for every code but 1MAD the second window's generator output comes
//         from the 32-bit funnel word by two multiply-adds, which moves work
//         from the ALU to the FMA pipe), the code, two tcgen05.st of 32
//         columns, one arrival.
//   12-17 issuers: operand B of their chunks, then the chunks' MMAs.
//   18-21 epilogue: D of each run out of TMEM (then zeroed) into the row sums,
//         the block ticket and, for the completing CTA, the output transform.
//         Warp 18 allocates TMEM.
// mbarriers: ring full/empty, A full/empty (6 TMEM slots), B full (bulk
// copies), D full/empty (2 accumulators).  Every parity wait is on a barrier
// whose previous phase the waiting thread itself has seen complete, so no
// wait can mistake a phase two behind for the one it needs.  Every wait is
// bounded: on timeout the thread sets the CTA's abort flag and the call's
// status word, every role stops, the issuers wait (bounded) for their MMAs,
// and TMEM is freed.
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
using tc::RowWords;
using tc::smem_desc;
using tc::smem_u32;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tmem_alloc;
using tc::tmem_dealloc;
using tc::tmem_st_wait;

constexpr int kCT = 8;             // tile columns per chunk (128 input columns)
constexpr int kTeams = 3;          // decoder teams
constexpr int kDecWarps = 4 * kTeams;
constexpr int kIss0 = kDecWarps;       // first issuer warp
constexpr int kIssuers = 6;            // over all four SM sub-partitions
constexpr int kEpiWarp0 = kIss0 + kIssuers;  // four warps, one per TMEM lane quarter
constexpr int kWarps = kEpiWarp0 + 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kSlotCols = 64;      // TMEM columns of one A slot (8 tiles x 16 weights / 2)
constexpr int kACol = 64;          // A slots after the two D accumulators (<= 32 columns each)
constexpr int kConstCol = kACol + kIssuers * kSlotCols;  // 8 columns: the centring column
constexpr int kTmemCols = 512;
constexpr int kExtK = 16;          // operand-B K elements of the centring MMA
constexpr int kKext = kCT * 16;    // operand-B K elements of a chunk
constexpr int kMmas = kKext / 16;  // MMAs (K = 16) per chunk
constexpr int kMaxRing = 12;
constexpr int kSmemLimit = 227 * 1024;  // dynamic shared memory of one CTA
constexpr int kEpiBarrier = 2;     // named barriers (0 is __syncthreads)
constexpr int kMaxM = 32;
static_assert(kConstCol + 8 <= kTmemCols, "TMEM columns");
static_assert(kIssuers % kTeams == 0, "each A slot belongs to one decoder team");

template <int K, int CB, int NB>
struct MvCfg {
  // the byte-sum codes store 1024 + S and are centred by one more MMA
  static constexpr bool kCentred = byte_sum_code<CB>();
  static constexpr int kBSlotBytes = (kKext + kExtK) * NB * 2;  // a chunk + the centring block
  static constexpr int kChunkBytesB = kKext * NB * 2;
  static constexpr int kStripWords = kCT * 8 * K;  // one tile row of the chunk, dense as the tensor copy lands
  static constexpr int kRowWords = kStripWords;
  static constexpr int kChunkBytes = 8 * kRowWords * 4;
  // the code ring takes what the control block, the operand-B slots and the
  // output transpose buffer leave (1 KB kept spare); a multiple of the
  // number of teams, so that each slot belongs to one decoder team
  static constexpr int kRingRaw =
      (kSmemLimit - 1024 - kIssuers * kBSlotBytes - kMaxM * 128 * 4 - 1024) / kChunkBytes;
  static constexpr int kRingClamped = kRingRaw > kMaxRing ? kMaxRing : (kRingRaw < kTeams ? kTeams : kRingRaw);
  static constexpr int kRing = kRingClamped - kRingClamped % kTeams;
  static_assert(2 * NB <= kACol, "D accumulators");
};

struct MvShared {
  uint64_t ring_full[kMaxRing];
  uint64_t ring_empty[kMaxRing];
  uint64_t a_full[kIssuers];
  uint64_t a_empty[kIssuers];
  uint64_t b_full[kIssuers];
  uint64_t d_full[2];
  uint64_t d_empty[2];
  uint64_t mma_done[kIssuers];
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

// D[tmem] += A[tmem] x B[smem desc] (always accumulating: D starts zeroed).
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

// Tensor copy of one box of a 2-D map into shared memory, completion counted
// on an mbarrier (coordinates in elements: x innermost).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
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
  {
    int hi = p.count - 1;  // the last layer whose first unit is <= u
    while (li < hi) {
      const int mid = (li + hi + 1) >> 1;
      if (u >= p.l[mid].u_begin) li = mid; else hi = mid - 1;
    }
  }
  const int lu = u - p.l[li].u_begin;
  rb = lu / p.l[li].nkb;
  kc = lu - rb * p.l[li].nkb;
}

// CTA whose stream-K range holds unit u (ranges [c*U/G, (c+1)*U/G), G <= U).
__device__ __forceinline__ int owner(long long u, long long units, long long grid) {
  return static_cast<int>(((u + 1) * grid - 1) / units);
}

__device__ __forceinline__ void tmem_st16_zero(uint32_t taddr) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1};" ::"r"(taddr), "r"(0u)
      : "memory");
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

// One TMEM column: two consecutive weights of a row as binary16, the first
// in the lower half, from their generator outputs.
//   byte-sum codes: 1024 + S (the dp4a byte sum spliced into the mantissa of
//   1024), centred later by the centring MMA;
//   three-instruction codes: the defined weight lo + hi, rounded to nearest
//   even -- one packed add of the word's two halves (broadcast) per weight.
template <int CB>
__device__ __forceinline__ uint32_t pack_col(uint32_t g0, uint32_t g1) {
  if constexpr (byte_sum_code<CB>()) {
    const uint32_t d0 = __dp4a(summed_bytes<CB>(g0), 0x01010101u, 0x6400u);
    const uint32_t d1 = __dp4a(summed_bytes<CB>(g1), 0x01010101u, 0x6400u);
    return __byte_perm(d0, d1, 0x5410);
  } else {
    const uint32_t h0 = mask_xor_3inst(g0);
    const uint32_t h1 = mask_xor_3inst(g1);
    const __half2 a = *reinterpret_cast<const __half2*>(&h0);
    const __half2 b = *reinterpret_cast<const __half2*>(&h1);
    const __half2 w0 = __hadd2(__low2half2(a), __high2half2(a));  // (w0, w0)
    const __half2 w1 = __hadd2(__low2half2(b), __high2half2(b));  // (w1, w1)
    return __byte_perm(*reinterpret_cast<const uint32_t*>(&w0), *reinterpret_cast<const uint32_t*>(&w1), 0x5410);
  }
}

template <int K, int CB, int NB, bool FUSE>
__global__ void __launch_bounds__(kThreads, 1) mv_kernel(const __grid_constant__ MvParams p) {
  using Cfg = MvCfg<K, CB, NB>;
  constexpr int kRing = Cfg::kRing;
  constexpr int kTw = 8 * K;  // words per tile
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  MvShared& sh = *reinterpret_cast<MvShared*>(smem_raw);
  const size_t ctrl = (sizeof(MvShared) + 1023) & ~static_cast<size_t>(1023);
  // the code ring first (1024-aligned for the tensor copies), then the
  // operand-B slots and the output transpose buffer
  uint32_t* ring = reinterpret_cast<uint32_t*>(smem_raw + ctrl);
  unsigned char* bslots = smem_raw + ctrl + static_cast<size_t>(kRing) * Cfg::kChunkBytes;  // kIssuers slots
  float* zt = reinterpret_cast<float*>(bslots + kIssuers * Cfg::kBSlotBytes);  // [M][128]

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
  auto issue_chunk = [&](int seq, int u) {  // by lane 0
    int li, rb, kc;
    locate(p, u, li, rb, kc);
    const int slot = seq % kRing;
    mbar_arrive_expect_tx(&sh.ring_full[slot], Cfg::kChunkBytes);
    tma_load_2d(ring + static_cast<size_t>(slot) * (Cfg::kChunkBytes / 4), &p.l[li].codes_map, kc * 32 * K, rb * 8,
                &sh.ring_full[slot]);
  };
  if (warp == kEpiWarp0) tmem_alloc(&sh.tmem_base, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&sh.ring_full[i], 1);
      mbar_init(&sh.ring_empty[i], 4);  // one elected arrival per warp of the consuming team
    }
    for (int i = 0; i < kIssuers; ++i) {
      mbar_init(&sh.a_full[i], 4);  // the four warps of the decoding team
      mbar_init(&sh.a_empty[i], 1);
      mbar_init(&sh.b_full[i], 1);
      mbar_init(&sh.mma_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.d_full[i], kIssuers);
      mbar_init(&sh.d_empty[i], 4);
    }
    sh.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  // Both accumulators start at zero (the MMAs always accumulate), and the
  // centring column of the byte-sum codes holds A = -(1024 + centre) at K
  // elements 0 and 1, zero elsewhere.
  if (warp >= kEpiWarp0) {
    const uint32_t lanes = static_cast<uint32_t>((warp & 3) * 32) << 16;
    tmem_st16_zero(tmem + lanes + 0);
    if constexpr (NB > 16) tmem_st16_zero(tmem + lanes + 16);
    tmem_st16_zero(tmem + lanes + NB);
    if constexpr (NB > 16) tmem_st16_zero(tmem + lanes + NB + 16);
    if constexpr (Cfg::kCentred) {
      const uint32_t c2 =
          static_cast<uint32_t>(__half_as_ushort(__int2half_rn(-(1024 + byte_sum_centre<CB>())))) * 0x10001u;
      tmem_st8(tmem + lanes + kConstCol, c2);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < kDecWarps) {
    // ---- decoders ----------------------------------------------------------------
    const int quarter = warp & 3;
    const int team = warp >> 2;  // 0 .. kTeams-1
    // The team's lead lane (warp 4*team, lane 0) loads the team's codes: its
    // first kRing/kTeams chunks now, then at the start of each chunk s the
    // chunk s - kTeams + kRing, into the slot of chunk s - kTeams (which the
    // team has finished reading).  A separate producer warp beside the
    // decoders measured one copy per ~1300 cycles: it starved for issue.
    const bool lead = quarter == 0 && lane == 0;
    const int count = hi - lo;
    int fetched = team;  // the team's next chunk to load
    if (lead)
      for (; fetched < count && fetched < kRing; fetched += kTeams) issue_chunk(fetched, lo + fetched);
    int consumed = team;  // the team's next chunk to wait for
    const int row = quarter * 32 + lane;  // row within the 128-row block (TMEM lane)
    const int trow = row >> 4;
    const int rr = row & 15;
    const int q0 = (rr * K) >> 1;  // first word of the row's window, and its bit offset
    const uint32_t off = static_cast<uint32_t>((rr * K) & 1) * 16u;
    const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
    // the second window of a funnel word through the FMA pipe where the
    // code's other steps load the ALU more (every code but 1MAD)
    constexpr bool kLoByImad = CB != kCb1Mad;
    for (int u = lo + team, seq = team; u < hi; u += kTeams, seq += kTeams) {
      const int rslot = seq % kRing;
      if (lead && fetched < count && seq >= kTeams) {
        // the slot of chunk fetched - kRing = seq - kTeams has been read by all four warps
        const int prev = fetched - kRing;
        if (mbar_wait(&sh.ring_empty[prev % kRing], (prev / kRing) & 1)) {
          issue_chunk(fetched, lo + fetched);
          fetched += kTeams;
        } else {
          set_abort(sh);
        }
      }
      bool ok = mbar_wait(&sh.ring_full[rslot], (seq / kRing) & 1);
      if (ok) consumed = seq + kTeams;
      if (!ok) set_abort(sh);
      if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) break;
      const uint32_t* rw = ring + static_cast<size_t>(rslot) * (Cfg::kChunkBytes / 4) + trow * Cfg::kRowWords;
      const int aslot = seq % kIssuers;
      const int ause = seq / kIssuers;
      bool stop = false;
#pragma unroll
      for (int g = 0; g < 2; ++g) {  // two groups of four tiles, 32 TMEM columns each
        uint32_t raw[4][RowWords<K>::kRaw];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
#pragma unroll
          for (int i = 0; i < RowWords<K>::kRaw; ++i) {
            int idx = q0 + i;
            if (idx >= kTw) idx -= kTw;
            raw[t][i] = rw[(g * 4 + t) * kTw + idx];
          }
        }
        if (g == 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.ring_empty[rslot]);
        }
        uint32_t v[32];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          uint32_t gen[16];
          row_generate<K, CB, kLoByImad>(raw[t], off, gen);
#pragma unroll
          for (int c = 0; c < 16; c += 2) v[t * 8 + c / 2] = pack_col<CB>(gen[c], gen[c + 1]);
        }
        if (g == 0 && ause > 0) {
          // the MMAs of the slot's previous chunk (this team's, four back) are done
          ok = mbar_wait(&sh.a_empty[aslot], (ause - 1) & 1);
          if (!ok) set_abort(sh);
          if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) {
            stop = true;
            break;
          }
        }
        tmem_st32(tmem + lanes + kACol + aslot * kSlotCols + g * 32, v);
      }
      if (stop) break;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.a_full[aslot]);
    }
    tmem_st_wait();
    // Copies the team loaded but never read (an aborted call) must land
    // before the CTA exits; each slot's phases move only with this team.
    if (lead)
      for (int c = consumed; c < fetched; c += kTeams) mbar_wait(&sh.ring_full[c % kRing], (c / kRing) & 1);
  } else if (warp < kIss0 + kIssuers) {
    // ---- issuers: operand B, then the MMAs of chunks seq = i (mod 4) --------------------
    const int is = warp - kIss0;
    unsigned char* bs = bslots + static_cast<size_t>(is) * Cfg::kBSlotBytes;  // this issuer's slot
    {
      // rows M.. and the centring block's unused K elements stay zero
      uint4* bz = reinterpret_cast<uint4*>(bs);
      for (int i = lane; i < Cfg::kBSlotBytes / 16; i += 32) bz[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncwarp();
    // x, the signs and the operand images may be written by the preceding
    // grid on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int M = p.M;
    const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
    constexpr uint32_t idesc = idesc_f16<NB>();
    constexpr uint32_t kLbo = (NB / 8) * 128;  // next 8 K elements
    constexpr uint32_t kSbo = 128;             // next 8 rows of N
    const uint64_t bd = smem_desc(smem_u32(bs), kLbo, kSbo);
    const uint32_t at = tm + kACol + is * kSlotCols;
    bool bad = p.debug_stall != 0;  // test hook: no MMA is ever issued, so the waits on them run out
    int issued = 0;
    int run = 0;
    for (int u0 = lo; u0 < hi && !bad; ++run) {
      int li, rb, kc0;
      locate(p, u0, li, rb, kc0);
      const MvLayer& L = p.l[li];
      const int u1 = min(hi, u0 + (L.nkb - kc0));  // this run: units u0 .. u1-1
      const int db = run & 1;
      const uint32_t dt = tm + static_cast<uint32_t>(db * NB);
      // the epilogue has taken the run two back out of this accumulator (and zeroed it)
      if (run >= 2) {
        const bool okd = mbar_wait(&sh.d_empty[db], ((run >> 1) - 1) & 1);
        if (!okd) set_abort(sh);
        if (__any_sync(0xFFFFFFFFu, !okd || aborted(sh))) break;
      }
      // this issuer's chunks of the run: seq = u - lo = is (mod kIssuers)
      const int s0 = u0 - lo, s1 = u1 - lo;
      int seq = s0 + ((is - s0) % kIssuers + kIssuers) % kIssuers;
      bool mine = false;
      for (; seq < s1; seq += kIssuers) {
        const int kc = kc0 + (seq - s0);
        const int use = seq / kIssuers;
        float csum[2] = {0.f, 0.f};  // centring sums of this chunk, per batch row
        uint2 hv[2];
        if constexpr (FUSE) {
          // Load and rotate before waiting for the slot: the L2 latency of x
          // overlaps the MMAs still reading it.
          const int col = kc * kCT * 16 + 4 * lane;
          const uint2 sr = L.s_in != nullptr ? *reinterpret_cast<const uint2*>(L.s_in + col) : make_uint2(0u, 0u);
          uint2 xr[2];
#pragma unroll
          for (int b = 0; b < 2; ++b)
            xr[b] = b < M ? *reinterpret_cast<const uint2*>(L.x + static_cast<size_t>(b) * L.n + col)
                          : make_uint2(0u, 0u);
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            if (b < M) {  // warp-uniform
              float v[4] = {__low2float(*reinterpret_cast<const __half2*>(&xr[b].x)),
                            __high2float(*reinterpret_cast<const __half2*>(&xr[b].x)),
                            __low2float(*reinterpret_cast<const __half2*>(&xr[b].y)),
                            __high2float(*reinterpret_cast<const __half2*>(&xr[b].y))};
              if (L.s_in != nullptr) {
                v[0] *= __low2float(*reinterpret_cast<const __half2*>(&sr.x));
                v[1] *= __high2float(*reinterpret_cast<const __half2*>(&sr.x));
                v[2] *= __low2float(*reinterpret_cast<const __half2*>(&sr.y));
                v[3] *= __high2float(*reinterpret_cast<const __half2*>(&sr.y));
                fwht128_warp(v, lane);
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
              }
              const __half2 o01 = __floats2half2_rn(v[0], v[1]);
              const __half2 o23 = __floats2half2_rn(v[2], v[3]);
              hv[b].x = *reinterpret_cast<const uint32_t*>(&o01);
              hv[b].y = *reinterpret_cast<const uint32_t*>(&o23);
              if constexpr (Cfg::kCentred)
                csum[b] = (__low2float(o01) + __high2float(o01)) + (__low2float(o23) + __high2float(o23));
            }
          }
        } else if constexpr (Cfg::kCentred) {
          // the chunk's sum of the binary16 operand values, from the image kernel
          if (lane < M) csum[0] = __ldcg(L.bsum + static_cast<size_t>(lane) * (L.n / kRowBlock) + kc);
        }
        // wait until this issuer's MMAs of its previous chunk are done with the slots
        bool ok = true;
        if (use > 0) ok = mbar_wait(&sh.a_empty[is], (use - 1) & 1);
        if (!ok) set_abort(sh);
        if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) {
          bad = true;
          break;
        }
        if constexpr (!FUSE) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&sh.b_full[is], Cfg::kChunkBytesB);
            bulk_g2s(bs, L.bimg + static_cast<size_t>(kc) * kKext * NB, Cfg::kChunkBytesB, &sh.b_full[is]);
          }
        } else {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            if (b < M) {
              // K elements k = 4*lane .. +3: half a 16-byte core row
              const int k = 4 * lane;
              *reinterpret_cast<uint2*>(bs + ((k >> 3) * (NB / 8) + (b >> 3)) * 128 + (b & 7) * 16 + (k & 7) * 2) =
                  hv[b];
            }
          }
        }
        if constexpr (Cfg::kCentred) {
          // Sum of the chunk's operand values per batch row, as hi + lo in
          // binary16 at K elements kKext and kKext + 1 of the centring block.
          float sums[2] = {csum[0], csum[1]};
          if constexpr (FUSE) {
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int d = 16; d > 0; d >>= 1) sums[b] += __shfl_xor_sync(0xFFFFFFFFu, sums[b], d);
          }
          if (lane < M) {
            const float sv = FUSE ? (lane == 0 ? sums[0] : sums[1]) : sums[0];
            const __half h = __float2half_rn(sv);
            const __half l = __float2half_rn(sv - __half2float(h));
            *reinterpret_cast<__half2*>(bs + ((kKext >> 3) * (NB / 8) + (lane >> 3)) * 128 + (lane & 7) * 16) =
                __halves2half2(h, l);
          }
        }
        // generic-proxy stores, read by the tensor core (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if constexpr (!FUSE) ok = mbar_wait(&sh.b_full[is], use & 1);  // the bulk copy has landed
        // the decoders' A of this chunk
        ok = ok && mbar_wait(&sh.a_full[is], use & 1) && !aborted(sh);
        if (__any_sync(0xFFFFFFFFu, !ok)) {
          set_abort(sh);
          bad = true;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < kMmas; ++j) mma_f16_ts_acc(dt, at + 8 * j, bd + ((2u * j * kLbo) >> 4), idesc);
          if constexpr (Cfg::kCentred)  // the centring MMA
            mma_f16_ts_acc(dt, tm + kConstCol, bd + ((static_cast<uint32_t>(kKext / 8) * kLbo) >> 4), idesc);
          mma_commit(&sh.a_empty[is]);
        }
        __syncwarp();
        mine = true;
        ++issued;
      }
      if (bad) break;
      // this issuer is done with the run: its commit arrives once its MMAs
      // are complete (a plain arrival if it had no chunk in the run)
      if (lane == 0) {
        if (mine)
          mma_commit(&sh.d_full[db]);
        else
          mbar_arrive(&sh.d_full[db]);
      }
      __syncwarp();
      u0 = u1;
    }
    // every MMA this issuer started has completed before TMEM is freed
    if (issued > 0) {
      if (lane == 0) mma_commit(&sh.mma_done[is]);
      __syncwarp();
      mbar_wait(&sh.mma_done[is], 0);
    }
  } else {
    // ---- epilogue ---------------------------------------------------------------------
    // The row sums, counters and y may be in use by the preceding grid.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int ew = warp & 3;  // TMEM lane quarter
    const int et = tid - kEpiWarp0 * 32;
    const int row = ew * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(ew * 32) << 16;
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
        tc::tmem_ld16(tmem + lanes + db * NB, d16);
#pragma unroll
        for (int j = 0; j < 16; ++j) d[j] = d16[j];
        if constexpr (NB > 16) {
          tc::tmem_ld16(tmem + lanes + db * NB + 16, d16);
#pragma unroll
          for (int j = 0; j < 16; ++j) d[16 + j] = d16[j];
        }
      }
      // zero the accumulator for the run after next, then hand it back
      tmem_st16_zero(tmem + lanes + db * NB);
      if constexpr (NB > 16) tmem_st16_zero(tmem + lanes + db * NB + 16);
      tmem_st_wait();
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
  if (warp == kEpiWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && aborted(sh) && p.status != nullptr) atomicOr(p.status, 1u);
}

template <int K, int CB, int NB>
inline size_t mv_smem_bytes() {
  using Cfg = MvCfg<K, CB, NB>;
  const size_t ctrl = (sizeof(MvShared) + 1023) & ~static_cast<size_t>(1023);
  return ctrl + static_cast<size_t>(Cfg::kRing) * Cfg::kChunkBytes + static_cast<size_t>(kIssuers) * Cfg::kBSlotBytes +
         static_cast<size_t>(kMaxM) * 128 * 4;
}

template <int K, int CB, int NB, bool FUSE>
exl3_status launch_mv_t(const MvParams& p, int grid, cudaStream_t stream) {
  size_t smem = mv_smem_bytes<K, CB, NB>();
  // At least 116 KB so that a single CTA is resident per SM (it owns all 512
  // TMEM columns; a second CTA would wait in tcgen05.alloc).
  if (smem < 116 * 1024) smem = 116 * 1024;
  if (cudaFuncSetAttribute(mv_kernel<K, CB, NB, FUSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  if (cudaLaunchKernelEx(&cfg, mv_kernel<K, CB, NB, FUSE>, p) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

// N = 16 up to 16 batch rows, else 32; x-tilde computed in the kernel for M <= 2.
template <int K, int CB>
exl3_status launch_mv_cb(const MvParams& p, int grid, cudaStream_t stream) {
  if (p.M <= 2) return launch_mv_t<K, CB, 16, true>(p, grid, stream);
  if (p.M <= 16) return launch_mv_t<K, CB, 16, false>(p, grid, stream);
  return launch_mv_t<K, CB, 32, false>(p, grid, stream);
}

template <int K>
exl3_status launch_mv_dispatch(const MvParams& p, int codebook, int grid, cudaStream_t stream) {
  switch (codebook) {
    case kCb3Inst: return launch_mv_cb<K, kCb3Inst>(p, grid, stream);
    case kCb1Mad: return launch_mv_cb<K, kCb1Mad>(p, grid, stream);
    case kCbMcg: return launch_mv_cb<K, kCbMcg>(p, grid, stream);
    default: return launch_mv_cb<K, kCbMul1>(p, grid, stream);
  }
}

}  // namespace mv
}  // namespace exl3

#define EXL3_DEFINE_MV_LAUNCHER(KK)                                                                  \
  namespace exl3 {                                                                                   \
  exl3_status launch_mv_k##KK(const MvParams& p, int codebook, int grid, cudaStream_t stream) {      \
    return mv::launch_mv_dispatch<KK>(p, codebook, grid, stream);                                    \
  }                                                                                                  \
  }
