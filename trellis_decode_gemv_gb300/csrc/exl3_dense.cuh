// Dense tensor-core kernel of the prefill path (tcgen05, sm_103a): z = W-hat
// x-tilde for M batch rows, x-tilde in operand-B images of NB batch rows per
// tile (NB = 64, 128 or 256, the MMA's N).  Two ways to feed operand A:
//
//  * from images (K = 0 below): W-hat decoded once per call into binary16
//    operand-A images in HBM ("decode a block once and reuse it", "Trellis
//    Quantization" Part fourteen), copied stage by stage into shared memory;
//  * fused (K = 1..8): sixteen decode warps turn the packed codes of each
//    stage into a binary16 image directly in shared memory (the defined
//    weights, or for the byte-sum codes the exact centred byte sums with the
//    scale applied to z), so the decoded matrix never goes through HBM.
//
// Persistent, one CTA per SM.  A unit is one 128-row output block x one tile
// of NB batch rows, numbered with the tile fastest so that CTAs that run at
// the same time share their operand-A stream (or codes) in L2; CTA b takes
// work items b, b + gridDim.x, ...  Whole units come first; the units of the
// last partial round (all units when there are fewer than SMs) may be split in
// K so that they fill the SMs.  A whole unit's D (128 x NB fp32 in TMEM) is the
// finished z of its block: the epilogue applies the scale, the output signs
// and the 128-point FWHT and writes y.  A split item adds D to the fp32 row
// sums zacc [M][m], and the item that completes the block's sums (an arrival
// counter per block and tile) finishes it from zacc.
//
// Warp roles: warps 0-3 and 6-9 epilogue (TMEM lane quarter = warp % 4), warp
// 4 MMA issue and TMEM allocation (one lane issues), warp 5 producer (one lane:
// 1-D bulk copies of each stage's operand B, and of operand A from images),
// warps 10-25 (fused only) decode.  Stages are 64 input columns: 4 MMAs of
// 128 x NB x 16, both operands in shared memory in the canonical K-major
// no-swizzle layout, in a 192 KB ring.  D is double-buffered over 2 NB TMEM
// columns, so a unit's epilogue overlaps the next unit's MMAs.  Every mbarrier
// wait is bounded; on timeout the CTA sets its abort flag and the status
// word, every role stops, the producer waits (bounded) for its copies in
// flight and the MMA lane for its MMAs, TMEM is freed.
#pragma once

#include "exl3_tc.cuh"

namespace exl3 {
namespace dense {

using tc::bulk_g2s;
using tc::mbar_arrive;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::mma_commit;
using tc::smem_desc;
using tc::smem_u32;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tmem_alloc;
using tc::tmem_dealloc;
using tc::tmem_ld16;

// (Eight stages of 32 columns, each half an image, ran 1.6x slower: every
// stage costs a fixed handshake on the MMA side that two MMAs do not cover.)
constexpr int kStageK = 64;         // input columns per stage
constexpr int kPrefetch = 8;  // stages of operand A requested into L2 ahead of use
constexpr int kABytes = 128 * kStageK * 2;   // 16 KB
constexpr int kRingBytes = 192 * 1024;
constexpr int kMaxStages = 8;

// Batch rows per tile NB (the MMA's N: 64, 128 or 256): operand-B bytes per
// stage, the ring depth that fills 192 KB (4, 6 or 8 stages) and the TMEM
// columns of the double-buffered D.
template <int NB>
struct Shape {
  static_assert(NB == 64 || NB == 128 || NB == 256, "tile width");
  static constexpr int kBBytes = NB * kStageK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kRingBytes / kStageBytes;
  static constexpr int kTmemCols = 2 * NB;
  static_assert(kStages <= kMaxStages, "ring depth");
};

// Warp roles; K = 0 takes operand A from images, K > 0 decodes it.
constexpr int kMmaWarp = 4;
constexpr int kProdWarp = 5;
constexpr int kDecWarp0 = 10;
constexpr int kEpiWarps = 8;  // warps 0-3 and 6-9
constexpr int kEpiThreads = 32 * kEpiWarps;
template <int K>
struct Roles {
  // fused: kGroups groups of eight decode warps (one per tile row of a
  // stage), group g decoding the stages seq with seq % kGroups == g
  static constexpr int kGroups = 2;
  static constexpr int kDecodeWarps = K == 0 ? 0 : 8 * kGroups;
  static constexpr int kThreads = (kDecWarp0 + kDecodeWarps) * 32;
};
constexpr int kSlice = 32;          // batch columns per epilogue slice
constexpr int kEpiBarrier = 1;

struct DenseParams {
  const unsigned char* aimg;  // operand-A images (K = 0)
  const uint32_t* codes;      // packed codes (K > 0)
  const __half* bimg;
  const __half* scales;
  const __half* s_out;
  __half* y;
  float* zacc;
  uint32_t* cnt;
  uint32_t* status;
  float zscale;     // factor of z in the epilogue: the byte-sum codes' scale when fused, else 1
  int m, n, M;
  int tiles;        // ceil(M / NB)
  int full;         // work items 0 .. full - 1: whole (block, tile) units over all of K
  int rem;          // the units after those, each split in `split` K ranges
  int split;
  int units;        // work items: full + rem * split
  int debug_stall;  // test hook: the producer posts nothing
};

struct Unit {
  int rb, t, ks0, ks1;  // output block, batch tile, stage range [ks0, ks1)
  int split;            // K ranges of this (block, tile): 1 = the item finishes it
};

// Work item i.  Units (block, tile) are numbered tile fastest.  The first
// `full` items are whole units; the last partial round of units is split in
// K, split index major, so that the CTAs that run together still share
// operand-A streams.
__device__ __forceinline__ Unit unit_of(const DenseParams& p, int i, int nstage) {
  Unit w;
  int q, s;
  if (i < p.full) {
    q = i;
    s = 0;
    w.split = 1;
  } else {
    const int f = i - p.full;
    s = f / p.rem;
    q = p.full + (f - s * p.rem);
    w.split = p.split;
  }
  w.t = q % p.tiles;
  w.rb = q / p.tiles;
  w.ks0 = s * nstage / w.split;
  w.ks1 = (s + 1) * nstage / w.split;
  return w;
}

struct DenseShared {
  uint64_t full[kMaxStages];   // from images: A and B landed; fused: the decode warps' arrivals
  uint64_t bfull[kMaxStages];  // fused: operand B landed
  uint64_t empty[kMaxStages];
  uint64_t d_full[2];
  uint64_t d_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t epi_go;
  uint32_t fix_go;
  uint32_t last;
  alignas(16) float zt[kSlice * 128];  // a slice of D transposed to [batch][row]
};

__device__ __forceinline__ bool aborted(const DenseShared& sh) {
  return *reinterpret_cast<const volatile uint32_t*>(&sh.abort) != 0u;
}
__device__ __forceinline__ void set_abort(DenseShared& sh) { atomicOr(&sh.abort, 1u); }
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarrier), "n"(kEpiThreads) : "memory");
}

// Bulk prefetch of global memory into L2 (no completion to wait for).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Generic-proxy writes to shared memory made visible to the async proxy (the
// tensor core reads the decoded operand through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// D[tmem] (+)= A[smem desc] x B[smem desc], kind::f16, cta_group::1.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One batch row of a 128-row block, lane holding rows 4*lane .. 4*lane + 3:
// y = binary16(Hb(s_out (.) (scale (.) z))) (no transform without s_out).
__device__ __forceinline__ void finish_rows(const DenseParams& p, float4 z, const float (&sc)[4],
                                            const float (&so)[4], int lane, size_t b, int r0) {
  float v[4] = {z.x * sc[0], z.y * sc[1], z.z * sc[2], z.w * sc[3]};
  if (p.s_out != nullptr) {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] *= so[j];
    fwht128_warp(v, lane);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] *= kInvSqrt128;
  }
  const __half2 o01 = __floats2half2_rn(v[0], v[1]);
  const __half2 o23 = __floats2half2_rn(v[2], v[3]);
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&o01);
  o.y = *reinterpret_cast<const uint32_t*>(&o23);
  *reinterpret_cast<uint2*>(p.y + b * p.m + r0) = o;
}

// Decode warp (d, g) of the fused kernel: tile row d of the 128-row block of
// every kGroups-th stage (stages g, g + kGroups, ...), 4 tiles of 16 columns.
// Lane (jt, pp) = (lane / 8, lane % 8) decodes rows 2pp and 2pp + 1 of tile
// jt (32 consecutive steps of the tile's stream) into the stage's operand-A
// image: 16 bytes of a row per store, row r of the block at (column group) *
// 2048 + r * 16.  Lanes with pp >= 4 store
// their second row first, so the eight lanes of each store phase cover all 32
// banks.  The code words of the next kAhead stages are in flight (registers)
// while a stage decodes: one stage's decode is shorter than an L2 round trip.
constexpr int kAhead = 2;

// Operand-A values of the fused kernel for two states, packed (s0 in the low
// half).  3INST and MCG: the defined binary16 weights.  1MAD and mul1: the
// centred byte sums S - centre, exact in binary16 (|S - centre| <= 510), with
// the code's binary32 scale applied to z in the epilogue instead (as the
// warp-shuffle kernel takes it from x): one dp4a puts S into the mantissa of
// binary16 1024 (bits 0x6400), one byte permute pairs the two, one packed
// subtraction removes 1024 + centre -- the int-to-half splice of "Trellis
// Quantization" Part three.
template <int CB>
__device__ __forceinline__ uint32_t fused_a_pair(uint32_t s0, uint32_t s1) {
  if constexpr (byte_sum_code<CB>()) {
    const uint32_t h0 = __dp4a(summed_bytes<CB>(generate<CB>(s0)), 0x01010101u, 0x6400u);
    const uint32_t h1 = __dp4a(summed_bytes<CB>(generate<CB>(s1)), 0x01010101u, 0x6400u);
    const uint32_t pr = __byte_perm(h0, h1, 0x5410);
    const __half c = __ushort_as_half(static_cast<unsigned short>(0x6400 + byte_sum_centre<CB>()));
    const __half2 w = __hsub2(*reinterpret_cast<const __half2*>(&pr), __half2half2(c));
    return *reinterpret_cast<const uint32_t*>(&w);
  } else {
    return decode_pair<CB>(s0, s1);
  }
}

struct StageCursor {
  int li, ks;
  Unit w;
};

template <int NB, int K, int CB>
__device__ __forceinline__ void decode_role(const DenseParams& p, DenseShared& sh, unsigned char* ring,
                                            int d, int g, int lane, int my_units, int nstage) {
  using S = Shape<NB>;
  constexpr int kGroups = Roles<K>::kGroups;
  constexpr int kStages = S::kStages;
  constexpr int kWords = RowPair<K>::kPairWords;
  const int jt = lane >> 3;
  const int pp = lane & 7;
  const int sw = (pp >> 2) & 1;
  const int tpr = p.n / 16;
  // byte offsets in an A image: first and second stored row, column groups 2jt and 2jt + 1
  const uint32_t o_first = static_cast<uint32_t>((2 * jt) * 2048 + d * 256 + (2 * pp + sw) * 16);
  const uint32_t o_second = static_cast<uint32_t>((2 * jt) * 2048 + d * 256 + (2 * pp + 1 - sw) * 16);
  const uint32_t ring_s = smem_u32(ring);
  if (my_units == 0) return;
  int total = 0;  // stages of all this CTA's work items
  for (int li = 0; li < my_units; ++li) {
    const Unit w = unit_of(p, static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x), nstage);
    total += w.ks1 - w.ks0;
  }
  // load cursor: the next stage of this warp whose words are not requested yet
  StageCursor c;
  c.li = 0;
  c.w = unit_of(p, static_cast<int>(blockIdx.x), nstage);
  c.ks = c.w.ks0;
  auto advance = [&]() {
    if (++c.ks >= c.w.ks1 && ++c.li < my_units) {
      c.w = unit_of(p, static_cast<int>(blockIdx.x) + c.li * static_cast<int>(gridDim.x), nstage);
      c.ks = c.w.ks0;
    }
  };
  for (int i = 0; i < g && i < total; ++i) advance();
  int requested = g;  // stage index of the cursor
  auto request = [&](uint32_t (&dst)[kWords]) {
    if (requested < total) {
      const uint32_t* t =
          p.codes + (static_cast<size_t>(c.w.rb * 8 + d) * tpr + static_cast<size_t>(c.ks) * 4 + jt) * (8 * K);
      load_row_pair<K>(t, pp, dst);
      requested += kGroups;
      for (int i = 0; i < kGroups; ++i) advance();
    }
  };
  uint32_t q[kAhead + 1][kWords];  // q[i]: the words of this warp's i-th next stage
#pragma unroll
  for (int i = 0; i < kAhead; ++i) request(q[i]);
  for (int seq = g; seq < total; seq += kGroups) {
    request(q[kAhead]);
    uint32_t st[32];
    pair_states<K>(q[0], st);
    uint32_t pk[16];  // row 2pp: pk[0..7], row 2pp + 1: pk[8..15], two weights per word
#pragma unroll
    for (int i = 0; i < 32; i += 2) pk[i / 2] = fused_a_pair<CB>(st[i], st[i + 1]);
    const int slot = seq % kStages;
    const int use = seq / kStages;
    const bool ok = use == 0 || mbar_wait(&sh.empty[slot], (use - 1) & 1);
    if (!ok) set_abort(sh);
    if (__any_sync(0xFFFFFFFFu, !ok || aborted(sh))) break;
    const uint32_t a = ring_s + static_cast<uint32_t>(slot * S::kStageBytes);
    // first stored row: row 2pp + sw
    const uint32_t f0 = sw ? pk[8] : pk[0], f1 = sw ? pk[9] : pk[1], f2 = sw ? pk[10] : pk[2],
                   f3 = sw ? pk[11] : pk[3];
    const uint32_t f4 = sw ? pk[12] : pk[4], f5 = sw ? pk[13] : pk[5], f6 = sw ? pk[14] : pk[6],
                   f7 = sw ? pk[15] : pk[7];
    const uint32_t g0 = sw ? pk[0] : pk[8], g1 = sw ? pk[1] : pk[9], g2 = sw ? pk[2] : pk[10],
                   g3 = sw ? pk[3] : pk[11];
    const uint32_t g4 = sw ? pk[4] : pk[12], g5 = sw ? pk[5] : pk[13], g6 = sw ? pk[6] : pk[14],
                   g7 = sw ? pk[7] : pk[15];
    st_shared_v4(a + o_first, f0, f1, f2, f3);
    st_shared_v4(a + o_first + 2048, f4, f5, f6, f7);
    st_shared_v4(a + o_second, g0, g1, g2, g3);
    st_shared_v4(a + o_second + 2048, g4, g5, g6, g7);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.full[slot]);
#pragma unroll
    for (int i = 0; i < kAhead; ++i)
#pragma unroll
      for (int j = 0; j < kWords; ++j) q[i][j] = q[i + 1][j];
  }
}

template <int NB, int K, int CB>
__global__ void __launch_bounds__(Roles<K>::kThreads, 1) dense_kernel(const DenseParams p) {
  using S = Shape<NB>;
  constexpr int kStages = S::kStages;
  constexpr int kStageBytes = S::kStageBytes;
  constexpr int kBBytes = S::kBBytes;
  constexpr bool kFused = K > 0;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  DenseShared& sh = *reinterpret_cast<DenseShared*>(smem_raw);
  const size_t ctrl = (sizeof(DenseShared) + 1023) & ~static_cast<size_t>(1023);
  unsigned char* ring = smem_raw + ctrl;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nstage = p.n / kStageK;
  const int my_units = p.units > static_cast<int>(blockIdx.x)
                           ? (p.units - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                           : 0;

  if (warp == kMmaWarp) tmem_alloc(&sh.tmem_base, S::kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.full[i], kFused ? 8 : 1);
      mbar_init(&sh.bfull[i], 1);
      mbar_init(&sh.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.d_full[i], 1);
      mbar_init(&sh.d_empty[i], kEpiThreads);
    }
    mbar_init(&sh.mma_done, 1);
    sh.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp >= kDecWarp0) {
    if constexpr (kFused)
      decode_role<NB, K, CB>(p, sh, ring, (warp - kDecWarp0) & 7, (warp - kDecWarp0) >> 3, lane, my_units, nstage);
  } else if (warp == kProdWarp) {
    // ---- producer: operand B (and A from images) of every stage into the ring ----------
    // With the failure-detection test hook set this warp posts nothing, so the
    // MMA lane's bounded wait for its operands runs out.
    if (lane == 0 && p.debug_stall == 0) {
      // Fused: the codes of a unit, one tile-row strip of its K range at a
      // time, are requested into L2 a unit ahead of the decode warps.
      auto prefetch_codes = [&](int li) {
        if (kFused && li < my_units) {
          const Unit w = unit_of(p, static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x), nstage);
          const size_t tpr = static_cast<size_t>(p.n / 16);
          for (int d = 0; d < 8; ++d)
            bulk_prefetch_l2(p.codes + (static_cast<size_t>(w.rb * 8 + d) * tpr + static_cast<size_t>(w.ks0) * 4) *
                                           (8 * K),
                             static_cast<uint32_t>(w.ks1 - w.ks0) * 128u * K);
        }
      };
      prefetch_codes(0);
      // The operand images are written by the preceding kernels on the stream.
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int seq = 0;
      bool stop = false;
      for (int li = 0; li < my_units && !stop; ++li) {
        const Unit w = unit_of(p, static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x), nstage);
        const unsigned char* a_src = kFused ? nullptr : p.aimg + static_cast<size_t>(w.rb) * nstage * kABytes;
        const __half* b_src = p.bimg + static_cast<size_t>(w.t) * NB * p.n;
        prefetch_codes(li + 1);
        for (int ks = w.ks0; ks < w.ks1; ++ks, ++seq) {
          const int slot = seq % kStages;
          const int use = seq / kStages;
          if (use > 0 && !mbar_wait(&sh.empty[slot], (use - 1) & 1)) set_abort(sh);
          if (aborted(sh)) {
            stop = true;
            break;
          }
          unsigned char* dst = ring + static_cast<size_t>(slot) * kStageBytes;
          uint64_t* bar = kFused ? &sh.bfull[slot] : &sh.full[slot];
          if constexpr (kFused) {
            mbar_arrive_expect_tx(bar, kBBytes);
          } else {
            mbar_arrive_expect_tx(bar, kStageBytes);
            bulk_g2s(dst, a_src + static_cast<size_t>(ks) * kABytes, kABytes, bar);
          }
          bulk_g2s(dst + kABytes, b_src + static_cast<size_t>(ks) * NB * kStageK, kBBytes, bar);
          // operand A streams from DRAM: ask for it kPrefetch stages before
          // the ring does, so that the ring's copies find it in L2
          if (!kFused && ks + kPrefetch < w.ks1)
            bulk_prefetch_l2(a_src + static_cast<size_t>(ks + kPrefetch) * kABytes, kABytes);
        }
      }
      // Wait (bounded) for the copies in flight.
      for (int i = 0; i < kStages && i < seq; ++i) {
        const int s = seq - 1 - i;
        mbar_wait(kFused ? &sh.bfull[s % kStages] : &sh.full[s % kStages], (s / kStages) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issue: the warp runs the loop, lane 0 issues ------------------------------
    constexpr uint32_t idesc = tc::idesc_f16<NB>();
    constexpr uint32_t kALbo = 16 * 128;         // next 8 K-elements of A (16 groups of 8 rows)
    constexpr uint32_t kBLbo = (NB / 8) * 128;  // next 8 K-elements of B
    const uint64_t adesc0 = smem_desc(smem_u32(ring), kALbo, 128);
    const uint64_t bdesc0 = smem_desc(smem_u32(ring + kABytes), kBLbo, 128);
    const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
    int seq = 0;
    bool bad = false;
    for (int li = 0; li < my_units && !bad; ++li) {
      const int db = li & 1;
      const bool okd = li < 2 || mbar_wait(&sh.d_empty[db], ((li >> 1) - 1) & 1);
      if (__any_sync(0xFFFFFFFFu, !okd)) {
        set_abort(sh);
        break;
      }
      tc_fence_after();
      const uint32_t dt = tm + static_cast<uint32_t>(NB * db);
      const Unit w = unit_of(p, static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x), nstage);
      for (int ks = w.ks0; ks < w.ks1; ++ks, ++seq) {
        const int slot = seq % kStages;
        const uint32_t par = (seq / kStages) & 1;
        const bool ok = mbar_wait(&sh.full[slot], par) && (!kFused || mbar_wait(&sh.bfull[slot], par)) &&
                        !aborted(sh);
        if (__any_sync(0xFFFFFFFFu, !ok)) {
          set_abort(sh);
          bad = true;
          break;
        }
        tc_fence_after();
        const uint32_t off = (static_cast<uint32_t>(slot) * kStageBytes) >> 4;
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < kStageK / 16; ++j)
            mma_f16_ss(dt, adesc0 + off + ((2u * j * kALbo) >> 4), bdesc0 + off + ((2u * j * kBLbo) >> 4), idesc,
                       (ks > w.ks0 || j > 0) ? 1u : 0u);
          mma_commit(&sh.empty[slot]);
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
    // ---- epilogue: D -> scale, output signs, FWHT -> y ---------------------------------
    // Eight warps: warp w reads TMEM lanes 32 * (w % 4) .. + 31 (rows of the
    // block); the two warps of a lane quarter take 16 batch columns each of a
    // 32-column slice.  Then every warp finishes whole batch rows.
    const int quarter = warp & 3;
    const int half = warp >= 6 ? 1 : 0;
    const int e = warp < 4 ? warp : warp - 2;  // epilogue warp index 0..7
    const int row = quarter * 32 + lane;       // TMEM lane = row of the 128-row block
    for (int li = 0; li < my_units; ++li) {
      if (tid == 0) sh.epi_go = aborted(sh) ? 0u : 1u;
      epi_sync();
      if (sh.epi_go == 0u) break;
      const Unit w = unit_of(p, static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x), nstage);
      const int rb = w.rb;
      const int t = w.t;
      const int rows = p.M - t * NB < NB ? p.M - t * NB : NB;  // batch rows of this tile
      const bool finish = w.split == 1;
      const int db = li & 1;
      const bool ok = !aborted(sh) && mbar_wait(&sh.d_full[db], (li >> 1) & 1);
      if (!ok) set_abort(sh);
      const bool warp_ok = !__any_sync(0xFFFFFFFFu, !ok);
      if (warp_ok) tc_fence_after();
      const int r0 = rb * kRowBlock + 4 * lane;  // this lane's four output rows in the FWHT
      float sc[4], so[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const uint2 sr = *reinterpret_cast<const uint2*>(p.scales + r0);
        const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
        const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
        sc[0] = __low2float(s01) * p.zscale;
        sc[1] = __high2float(s01) * p.zscale;
        sc[2] = __low2float(s23) * p.zscale;
        sc[3] = __high2float(s23) * p.zscale;
      }
      if (p.s_out != nullptr) {
        const uint2 sr = *reinterpret_cast<const uint2*>(p.s_out + r0);
        const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
        const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
        so[0] = __low2float(s01);
        so[1] = __high2float(s01);
        so[2] = __low2float(s23);
        so[3] = __high2float(s23);
      }
      const int slices = (rows + kSlice - 1) / kSlice;
#pragma unroll 1
      for (int sl = 0; sl < slices; ++sl) {
        const int b0 = sl * kSlice + 16 * half;
        if (warp_ok && b0 < rows) {  // warp-uniform
          float dv[16];
          tmem_ld16(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(NB * db + b0), dv);
#pragma unroll
          for (int j = 0; j < 16; ++j) sh.zt[(16 * half + j) * kRowBlock + row] = dv[j];
        }
        epi_sync();
        if (!__any_sync(0xFFFFFFFFu, aborted(sh))) {  // warp-uniform: the FWHT shuffles
          // one batch row per warp at a time: lane holds rows 4*lane .. +3
          const int nb = rows - sl * kSlice < kSlice ? rows - sl * kSlice : kSlice;
#pragma unroll 4
          for (int bl = e; bl < nb; bl += kEpiWarps) {
            const float4 z = *reinterpret_cast<const float4*>(&sh.zt[bl * kRowBlock + 4 * lane]);
            const size_t b = static_cast<size_t>(t) * NB + sl * kSlice + bl;
            if (finish)
              finish_rows(p, z, sc, so, lane, b, r0);
            else
              atomicAdd(reinterpret_cast<float4*>(p.zacc + b * p.m + r0), z);
          }
        }
        epi_sync();  // zt is rewritten by the next slice
      }
      if (warp_ok) tc_fence_before();
      mbar_arrive(&sh.d_empty[db]);
      if (finish) continue;
      // K split: the unit whose partial sums complete the block finishes it
      // from zacc (read through L2) and leaves zacc and the counter at zero.
      if (tid == 0) sh.fix_go = aborted(sh) ? 0u : 1u;
      epi_sync();
      if (sh.fix_go == 0u) continue;
      __threadfence();
      epi_sync();
      uint32_t* cnt = p.cnt + static_cast<size_t>(rb) * p.tiles + t;
      if (tid == 0) sh.last = atomicAdd(cnt, 1u) == static_cast<uint32_t>(w.split - 1) ? 1u : 0u;
      epi_sync();
      if (sh.last == 0u) continue;
      __threadfence();
      // kFixRows batch rows per warp in flight: the loads are L2 round trips
      constexpr int kFixRows = kFused ? 4 : 8;
#pragma unroll 1
      for (int b0 = e; b0 < rows; b0 += kEpiWarps * kFixRows) {
        float4 z[kFixRows];
#pragma unroll
        for (int i = 0; i < kFixRows; ++i) {
          const int bl = b0 + kEpiWarps * i;
          z[i] = bl < rows ? __ldcg(reinterpret_cast<const float4*>(
                                 p.zacc + (static_cast<size_t>(t) * NB + bl) * p.m + r0))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kFixRows; ++i) {
          const int bl = b0 + kEpiWarps * i;
          if (bl >= rows) break;  // warp-uniform
          const size_t b = static_cast<size_t>(t) * NB + bl;
          __stcg(reinterpret_cast<float4*>(p.zacc + b * p.m + r0), make_float4(0.f, 0.f, 0.f, 0.f));
          finish_rows(p, z[i], sc, so, lane, b, r0);
        }
      }
      if (tid == 0) *cnt = 0u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, S::kTmemCols);
  }
  if (tid == 0 && aborted(sh) && p.status != nullptr) atomicOr(p.status, 1u);
}

// Launch over all SMs (fewer when there are fewer work items), with
// programmatic stream serialization: the kernel starts while its predecessor
// finishes and waits for it before reading operand B.  p.tiles, p.full,
// p.rem, p.units are filled in here from p.M and split.
template <int NB, int K, int CB>
exl3_status launch_dense_kernel(DenseParams p, int split, cudaStream_t stream) {
  using S = Shape<NB>;
  p.tiles = (p.M + NB - 1) / NB;
  const int units = (p.m / kRowBlock) * p.tiles;
  const int sms = device_sm_count();
  p.split = split;
  p.rem = split > 1 ? units % sms : 0;
  p.full = units - p.rem;
  p.units = p.full + p.rem * split;
  const size_t ctrl = (sizeof(DenseShared) + 1023) & ~static_cast<size_t>(1023);
  const size_t smem = ctrl + static_cast<size_t>(S::kStages) * S::kStageBytes;
  if (cudaFuncSetAttribute(dense_kernel<NB, K, CB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return EXL3_ERR_CUDA;
  int grid = sms;
  if (grid > p.units) grid = p.units;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Roles<K>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, dense_kernel<NB, K, CB>, p) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

// The fused kernel for K-bit codes: NB in {64, 128, 256}, any codebook.
template <int K>
exl3_status launch_fused_dispatch(const DenseParams& p, int codebook, int nb, int split, cudaStream_t stream) {
  if (nb == 64) {
    switch (codebook) {
      case kCb3Inst: return launch_dense_kernel<64, K, kCb3Inst>(p, split, stream);
      case kCb1Mad: return launch_dense_kernel<64, K, kCb1Mad>(p, split, stream);
      case kCbMcg: return launch_dense_kernel<64, K, kCbMcg>(p, split, stream);
      default: return launch_dense_kernel<64, K, kCbMul1>(p, split, stream);
    }
  }
  if (nb == 128) {
    switch (codebook) {
      case kCb3Inst: return launch_dense_kernel<128, K, kCb3Inst>(p, split, stream);
      case kCb1Mad: return launch_dense_kernel<128, K, kCb1Mad>(p, split, stream);
      case kCbMcg: return launch_dense_kernel<128, K, kCbMcg>(p, split, stream);
      default: return launch_dense_kernel<128, K, kCbMul1>(p, split, stream);
    }
  }
  if (nb == 256) {
    switch (codebook) {
      case kCb3Inst: return launch_dense_kernel<256, K, kCb3Inst>(p, split, stream);
      case kCb1Mad: return launch_dense_kernel<256, K, kCb1Mad>(p, split, stream);
      case kCbMcg: return launch_dense_kernel<256, K, kCbMcg>(p, split, stream);
      default: return launch_dense_kernel<256, K, kCbMul1>(p, split, stream);
    }
  }
  return EXL3_ERR_SHAPE;
}

}  // namespace dense

// One translation unit per K (exl3_fused_k<K>.cu).
exl3_status launch_fused_k1(const dense::DenseParams& p, int codebook, int nb, int split, cudaStream_t stream);
exl3_status launch_fused_k2(const dense::DenseParams& p, int codebook, int nb, int split, cudaStream_t stream);
exl3_status launch_fused_k3(const dense::DenseParams& p, int codebook, int nb, int split, cudaStream_t stream);
exl3_status launch_fused_k4(const dense::DenseParams& p, int codebook, int nb, int split, cudaStream_t stream);
exl3_status launch_fused_k5(const dense::DenseParams& p, int codebook, int nb, int split, cudaStream_t stream);
exl3_status launch_fused_k6(const dense::DenseParams& p, int codebook, int nb, int split, cudaStream_t stream);
exl3_status launch_fused_k7(const dense::DenseParams& p, int codebook, int nb, int split, cudaStream_t stream);
exl3_status launch_fused_k8(const dense::DenseParams& p, int codebook, int nb, int split, cudaStream_t stream);

}  // namespace exl3

#define EXL3_DEFINE_FUSED_LAUNCHER(KK)                                                                  \
  namespace exl3 {                                                                                      \
  exl3_status launch_fused_k##KK(const dense::DenseParams& p, int codebook, int nb, int split,           \
                                 cudaStream_t stream) {                                                  \
    return dense::launch_fused_dispatch<KK>(p, codebook, nb, split, stream);                             \
  }                                                                                                     \
  }
