// Host-side helpers of libexl3: argument validation, launch plans and the
// internal launcher declarations shared by the translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/exl3.h"

namespace exl3 {

constexpr int kRowBlock = 128;      // rows per output block (one output FWHT)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline exl3_status check_shape(int m, int n) {
  if (m <= 0 || n <= 0 || (m % kRowBlock) != 0 || (n % kRowBlock) != 0) return EXL3_ERR_SHAPE;
  return EXL3_OK;
}

// floor(u / d) for 0 <= u < n_end as the high word of u * magic, with magic =
// ceil(2^32 / d): u * magic / 2^32 = u / d + u * e / (d * 2^32), e = magic * d
// - 2^32 < d, so the floor is exact while u * e < 2^32.  0 when that does not
// hold for every u < n_end (or d < 2): the caller divides.
inline uint32_t div_magic(long long d, long long n_end) {
  if (d < 2 || d >= (1LL << 32)) return 0;
  const unsigned long long m = ((1ULL << 32) + static_cast<unsigned long long>(d) - 1) / static_cast<unsigned long long>(d);
  const unsigned long long e = m * static_cast<unsigned long long>(d) - (1ULL << 32);
  if (n_end < 0 || n_end >= (1LL << 32)) return 0;
  return static_cast<unsigned long long>(n_end) * e < (1ULL << 32) ? static_cast<uint32_t>(m) : 0u;
}

inline exl3_status check_k_cb(int K, int codebook) {
  if (K < 1 || K > 8) return EXL3_ERR_K;
  if (codebook < EXL3_CB_3INST || codebook > EXL3_CB_MUL1) return EXL3_ERR_CODEBOOK;
  return EXL3_OK;
}

inline exl3_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? EXL3_OK : EXL3_ERR_CUDA;
}

// Number of SMs of the current device (queried once per device).
int device_sm_count();

// Workspace layout (all offsets 256-byte aligned):
//   counters  one uint32 per 128-row block, then one status word (non-zero
//             after a device-side wait of the tensor-core kernel timed out);
//   zacc      fp32 [M][m]: row sums accumulated by the layer kernels;
//   bimg      binary16: the rotated x laid out as the tensor-core kernel's
//             operand B, one (tc_nb(M) x 128) image per 128 input columns;
//   bsum      fp32 [M][n/128]: sums of the binary16 rotated x per 128 block
//             (1MAD correction of the tensor-core kernel).
// counters and zacc must be zero before a call and are zero after it.
inline size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }
// Batch columns of the tensor-core MMAs (N of the 128 x N x 16 shape).
inline int tc_nb(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : 128; }
// Batch rows per pass of exl3_gemm above EXL3_MAX_BATCH (the N = 128 kernel).
constexpr int kPrefillRows = 128;
inline size_t counters_bytes(int m) {
  return align256(sizeof(uint32_t) * (static_cast<size_t>(m / kRowBlock) + 1));
}
inline size_t zacc_offset(int m) { return counters_bytes(m); }
inline size_t bimg_offset(int m, int M) {
  return zacc_offset(m) + align256(sizeof(float) * static_cast<size_t>(M) * m);
}
inline size_t bsum_offset(int m, int n, int M) {
  return bimg_offset(m, M) + align256(sizeof(__half) * static_cast<size_t>(tc_nb(M)) * n);
}
inline size_t workspace_total(int m, int n, int M) {
  return bsum_offset(m, n, M) + align256(sizeof(float) * static_cast<size_t>(M) * (n / kRowBlock));
}

// Launch plan of the warp-shuffle path.  Layers with at least 1024 tiles per
// SM (and any batch chunk above 2) use the sub-unit kernel: one CTA per SM
// (fewer for tiny layers) and sub-units of S in {16, 8, 4} tiles, the largest
// that still gives every warp about two sub-units.  Smaller layers at batch
// chunks of 1 or 2 use the segment kernel (sub = 0): one wave of 5 or 4
// 256-thread CTAs per SM, at least 4 tile columns of work per CTA.
struct LayerPlan {
  int ctas;
  int sub;  // 0: segment kernel
};
LayerPlan plan_layer(int m, int n, int mb, int sm_count);

// ---- groups of independent layers (exl3_gemm_grouped) ---------------------------
constexpr int kMaxGroup = EXL3_MAX_GROUP;

// One layer of the sub-unit kernel.  Its sub-units are numbered from u_begin
// in the group's sequence, tile row major.
struct GroupLayer {
  const uint32_t* codes;
  const uint32_t* xdup;  // x pairs [mb][n]
  float* zacc;           // fp32 row sums [mb][m]
  int m, n;
  int u_begin;
  int per_row;           // sub-units per tile row
  uint32_t row_magic;    // div_magic(per_row, the layer's sub-units), 0: divide
};

struct GroupArgs {
  GroupLayer l[kMaxGroup];
  int count;
  int units;  // sub-units of all layers
  int sub;    // tiles per sub-unit
  int ctas;
  // the one-K kernel (launch_group_kset_k*): layers ordered by code, the
  // sub-units of code c end at code_end[c]
  int code_end[4];
};

// x pairs and output transforms of a group: one warp per (layer, batch row,
// 128-block); the jobs of layer i start at job_begin.
struct XdupEntry {
  const __half* x;      // [rows][n]
  const __half* s_in;   // [n] or nullptr
  uint32_t* xd;         // [rows][n]
  int n;
  float factor;         // the layer's code's x factor
  long long job_begin;
};
struct XdupGroup {
  XdupEntry e[kMaxGroup];
  int count;
  int rows;
  long long jobs;
};
// Operand-B images of the decode-MMA kernel for a group of layers: one warp
// per (layer, batch row, 128-block); the jobs of layer i start at job_begin.
struct BimgEntry {
  const __half* x;      // [M][n]
  const __half* s_in;   // [n] or nullptr
  __half* bimg;         // the images (mv_bimg_bytes(n, M))
  float* bsum;          // [M][n/128] block sums, or nullptr
  int n;
  long long job_begin;
};
struct BimgGroup {
  BimgEntry e[kMaxGroup];
  int count;
  int M;
  int nb;               // rows per image tile (16 or 32)
  long long jobs;
};
struct EpiEntry {
  float* zacc;            // [rows][m], zeroed after reading
  const __half* scales;   // [m]
  const __half* s_out;    // [m] or nullptr
  __half* y;              // [rows][m]
  int m;
  long long job_begin;
};
struct EpiGroup {
  EpiEntry e[kMaxGroup];
  int count;
  int rows;
  long long jobs;
};

struct LayerArgs {
  const uint32_t* codes;
  int K, codebook, m, n;
  const __half* s_in;
  const __half* s_out;
  const __half* scales;
  const __half* x;  // [mb][n]
  __half* y;        // [mb][m]
  float* zacc;        // [mb][m] fp32 row sums, zero on entry and exit
  uint32_t* counters;
  uint32_t* status;   // device-side error bits (tensor-core path), or nullptr
  const uint32_t* xdup;  // warp-shuffle kernel: x pairs [mb][n]
  int ctas;           // warp-shuffle kernel: grid size
  int sub;            // warp-shuffle kernel: tiles per sub-unit (32, 16, 8 or 4)
  int debug_stall;    // tensor-core kernel: test hook, post no operand B
};

// ---- decode-MMA kernel (csrc/exl3_mv.cuh), 1 <= M <= 32 -------------------------
// One layer of a call.  Units of layer i are u_begin .. u_begin + (m/128)*nkb.
struct MvLayer {
  // the codes as a 2-D tensor of 64-bit elements: (m/16) tile rows of
  // (n/16) * 4K elements; one box is the 8 tile-row strips of one chunk
  CUtensorMap codes_map;
  const uint32_t* codes;
  const __half* x;       // [M][n] (x warps compute x-tilde; M <= 2)
  const __half* s_in;    // [n] or nullptr
  const __half* bimg;    // operand-B images, nkb chunks of kKext x NB (M > 2)
  const float* bsum;     // [M][n/128] sums of the images' binary16 values (M > 2, byte-sum codes)
  const __half* scales;  // [m]
  const __half* s_out;   // [m] or nullptr
  __half* y;             // [M][m]
  float* zacc;           // [M][m] fp32 row sums, zero on entry and exit
  uint32_t* cnt;         // [m/128] arrival counters, zero on entry and exit
  int m, n;
  int u_begin;
  int nkb;               // chunks per 128-row block
};

struct MvParams {
  MvLayer l[kMaxGroup];
  int count;
  int units;
  int M;
  uint32_t* status;      // ORed with 1 when a bounded wait ran out
  int debug_stall;       // test hook: operand B is never posted
};

// The decode-MMA kernel works in chunks of 128 input columns; the byte-sum
// codes (1MAD, mul1) are centred through the sums of operand B.
inline bool mv_centred(int codebook) { return codebook == EXL3_CB_1MAD || codebook == EXL3_CB_MUL1; }
constexpr int kMvChunkCols = 128;
// Batch columns N of its MMAs.
inline int mv_nb(int M) { return M <= 16 ? 16 : 32; }
// Operand-B images of the decode-MMA kernel for M > 2 (x-tilde computed in
// the kernel below that): launch_bimg's layout, one (NB x 128) binary16
// K-major image per 128-column block.
inline size_t mv_bimg_bytes(int n, int M) { return sizeof(__half) * static_cast<size_t>(mv_nb(M)) * n; }
// ... and their block sums, fp32 [M][n/128].
inline size_t mv_bsum_bytes(int n, int M) { return sizeof(float) * static_cast<size_t>(M) * (n / kRowBlock); }
exl3_status launch_mv_k1(const MvParams& p, int codebook, int grid, cudaStream_t stream);
exl3_status launch_mv_k2(const MvParams& p, int codebook, int grid, cudaStream_t stream);
exl3_status launch_mv_k3(const MvParams& p, int codebook, int grid, cudaStream_t stream);
exl3_status launch_mv_k4(const MvParams& p, int codebook, int grid, cudaStream_t stream);
exl3_status launch_mv_k5(const MvParams& p, int codebook, int grid, cudaStream_t stream);
exl3_status launch_mv_k6(const MvParams& p, int codebook, int grid, cudaStream_t stream);
exl3_status launch_mv_k7(const MvParams& p, int codebook, int grid, cudaStream_t stream);
exl3_status launch_mv_k8(const MvParams& p, int codebook, int grid, cudaStream_t stream);
// A call of the decode-MMA kernel over p.count layers of K bits and the given
// code at batch p.M: fills the plan fields (units, chunks, grid), writes the
// operand images first for M > 2 (p.l[i].bimg must point at
// mv_bimg_bytes(n, M) of workspace each), then one launch.
exl3_status run_mv(MvParams p, int K, int codebook, cudaStream_t stream);
// Kernel launches of run_mv.
inline int mv_launches(int count, int M) { return M <= 2 || count < 1 ? 1 : 2; }

// The int8-activation layer kernel over a group of layers (a batch chunk of
// mb rows); each sub-unit looks up its layer, as in GroupArgs.
struct I8Layer {
  const uint32_t* codes;
  const int32_t* q4;     // [mb][n]: each int8 activation replicated into the four bytes of a word
  const int32_t* tcorr;  // [mb][n/16]: centre x (sum of the tile's 16 activations)
  const float* cs;       // [mb][n/128]: C x the block's activation scale
  float* zacc;           // [mb][m] fp32 row sums
  int m, n;
  int u_begin;  // first sub-unit of this layer
  int per_row;  // sub-units per tile row
  uint32_t row_magic;  // div_magic(per_row, the layer's sub-units), 0: divide
};
struct I8Args {
  I8Layer l[kMaxGroup];
  int count;
  int sub;  // tiles per sub-unit
  int ctas;
  long long units;  // sub-units of all layers
  // the one-K kernel (launch_i8_kset_k*): layers ordered by code, the
  // sub-units of 1MAD end at class_end[0], of mul1 at class_end[1]
  long long class_end[2];
};
// Batch 1, 32-tile sub-units: the 1MAD and mul1 layers of one K in one
// kernel, one loop per code (I8Args::class_end).
exl3_status launch_i8_kset_k1(const I8Args& a, cudaStream_t stream);
exl3_status launch_i8_kset_k2(const I8Args& a, cudaStream_t stream);
exl3_status launch_i8_kset_k3(const I8Args& a, cudaStream_t stream);
exl3_status launch_i8_kset_k4(const I8Args& a, cudaStream_t stream);
exl3_status launch_i8_kset_k5(const I8Args& a, cudaStream_t stream);
exl3_status launch_i8_kset_k6(const I8Args& a, cudaStream_t stream);
exl3_status launch_i8_kset_k7(const I8Args& a, cudaStream_t stream);
exl3_status launch_i8_kset_k8(const I8Args& a, cudaStream_t stream);
exl3_status launch_i8_k1(const I8Args& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_i8_k2(const I8Args& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_i8_k3(const I8Args& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_i8_k4(const I8Args& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_i8_k5(const I8Args& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_i8_k6(const I8Args& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_i8_k7(const I8Args& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_i8_k8(const I8Args& a, int codebook, int mb, cudaStream_t stream);

// Internal launchers (one translation unit per K for the layer kernels).
exl3_status launch_rht(const __half* in, const __half* signs, __half* out, int rows, int d,
                       cudaStream_t stream);
// Operand-B images of the tensor-core kernels: the M rows in tiles of nb; for
// tile t and every 128-column block kb of x-tilde = Hb(s_in (.) x) (x itself
// when s_in is NULL), the nb x 128 binary16 K-major image at bimg + t * nb * n
// + kb * nb * 128 (rows past M zero), and for bsum != NULL the fp32 sums
// bsum[b * (n/128) + kb] of the binary16 values.
exl3_status launch_bimg(const __half* x, const __half* s_in, __half* bimg, float* bsum, int M,
                        int nb, int n, cudaStream_t stream);
// x pairs of a group; codebook >= 0 sets every entry's x factor from it, -1
// keeps the factors the entries carry (layers of different codes).
exl3_status launch_xdup_group(XdupGroup g, int codebook, cudaStream_t stream);
// One launch of the operand-image kernel for every entry of g (nb < 128).
exl3_status launch_bimg_group(BimgGroup g, int M, int nb, cudaStream_t stream);
// The factor the x pairs carry for a code (the byte-sum codes' scale).
float code_x_factor(int codebook);

exl3_status launch_epi_group(EpiGroup g, cudaStream_t stream);
// The sub-unit kernel over a group (a.sub > 0 tiles per sub-unit, a.ctas CTAs).
// Batch 1, 32-tile sub-units: the layers of every code of one K in one
// kernel, one loop per code over that code's sub-units (GroupArgs::code_end).
exl3_status launch_group_kset_k1(const GroupArgs& a, cudaStream_t stream);
exl3_status launch_group_kset_k2(const GroupArgs& a, cudaStream_t stream);
exl3_status launch_group_kset_k3(const GroupArgs& a, cudaStream_t stream);
exl3_status launch_group_kset_k4(const GroupArgs& a, cudaStream_t stream);
exl3_status launch_group_kset_k5(const GroupArgs& a, cudaStream_t stream);
exl3_status launch_group_kset_k6(const GroupArgs& a, cudaStream_t stream);
exl3_status launch_group_kset_k7(const GroupArgs& a, cudaStream_t stream);
exl3_status launch_group_kset_k8(const GroupArgs& a, cudaStream_t stream);
exl3_status launch_group_k1(const GroupArgs& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_group_k2(const GroupArgs& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_group_k3(const GroupArgs& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_group_k4(const GroupArgs& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_group_k5(const GroupArgs& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_group_k6(const GroupArgs& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_group_k7(const GroupArgs& a, int codebook, int mb, cudaStream_t stream);
exl3_status launch_group_k8(const GroupArgs& a, int codebook, int mb, cudaStream_t stream);
// One layer through the tensor-core path (operand images, MMA kernel, output
// transform) or through the warp-shuffle path (batch chunks of 8/4/2/1; x pairs
// and the sub-unit kernel, or the segment kernel, then the output transform),
// with explicit workspace regions: fp32 row sums zacc [M][m] (zero on entry and
// exit), the status word, operand images bimg and block sums bsum (tensor), x
// pairs xd [8][n] (warp-shuffle).
exl3_status run_tensor(LayerArgs a, int M, float* zacc, uint32_t* status, __half* bimg, float* bsum,
                       cudaStream_t cs);
exl3_status run_shuffle(LayerArgs a, int M, float* zacc, uint32_t* xd, cudaStream_t cs);

// Sub-unit size S in {16, 8, 4} for `tiles` tiles at batch chunk mb: the
// largest that still gives every warp of the one CTA per SM about two
// sub-units.
int choose_sub(long long tiles, int mb, int sm_count);

// x pairs of the warp-shuffle kernel: for each of `rows` rows of x, x-tilde =
// Hb(s_in (.) x) (x without s_in) times the code's x factor (1 for 3INST,
// 1/sqrt(21845) for 1MAD), rounded to binary16 and duplicated into both halves
// of a 32-bit word, xd[row][n].  A programmatic dependent of the preceding
// kernel (waits for it before reading x).
exl3_status launch_xdup(const __half* x, const __half* s_in, uint32_t* xd, int rows, int n,
                        int codebook, cudaStream_t stream);
exl3_status launch_decode(const uint32_t* codes, int K, int codebook, int m, int n, __half* w,
                          cudaStream_t stream);
// W-hat decoded into the dense kernel's operand-A images (m * n binary16 in
// 16 KB images of 128 rows x 64 columns, canonical K-major layout).
exl3_status launch_decode_aimg(const uint32_t* codes, int K, int codebook, int m, int n,
                               unsigned char* aimg, cudaStream_t stream);
// Dense prefill kernel: z = A x-tilde for M batch rows, A from the operand-A
// images, x-tilde from operand-B images of nb rows per tile (nb = 64, 128 or
// 256; bimg + tile * nb * n halves), then y = binary16(Hb(s_out (.) (scale (.)
// z))).
// With split == 1 every work unit covers all of K and finishes its block from
// tensor memory; with split > 1 each unit covers 1/split of K and adds its
// partial z to zacc [M][m], and the unit that brings the block's counter
// cnt[block * tiles + tile] to split finishes the block from zacc and zeroes
// zacc and the counter.  debug_stall: the failure-detection test hook, post no
// operands.
exl3_status launch_dense(const unsigned char* aimg, const __half* bimg, const __half* scales,
                         const __half* s_out, __half* y, float* zacc, uint32_t* cnt, int m, int n, int M,
                         int nb, int split, uint32_t* status, int debug_stall, cudaStream_t stream);

// Fused prefill kernel: as launch_dense, but each CTA decodes operand A from
// the packed codes (K bits, codebook) into shared memory stage by stage; nb =
// 128 or 256.  No operand-A images.
exl3_status launch_fused(const uint32_t* codes, int K, int codebook, const __half* bimg, const __half* scales,
                         const __half* s_out, __half* y, float* zacc, uint32_t* cnt, int m, int n, int M,
                         int nb, int split, uint32_t* status, int debug_stall, cudaStream_t stream);

// Dense prefill path (exl3_gemm above EXL3_MAX_BATCH): batch rows per MMA tile
// (N of 128 x N x 16) and the workspace layout: counters and status as above,
// zacc fp32 [M][m], bimg one (nb x n) operand-B image per tile of nb batch
// rows, aimg the decoded matrix as m * n binary16 operand-A images, cnt one
// uint32 per (128-row block, tile): K-split arrivals.  The regions are sized
// for tiles of kDenseNB rows; a batch of M <= 128 rows runs as one tile of
// dense_nb(M) <= M rounded up, which fits in them.
constexpr int kDenseNB = 256;
inline int dense_nb(int M) { return M <= 64 ? 64 : M <= 128 ? 128 : kDenseNB; }
inline int dense_tiles(int M) { return (M + kDenseNB - 1) / kDenseNB; }
inline size_t dense_bimg_offset(int m, int M) { return bimg_offset(m, M); }
inline size_t dense_aimg_offset(int m, int n, int M) {
  return dense_bimg_offset(m, M) +
         align256(sizeof(__half) * static_cast<size_t>(dense_tiles(M)) * kDenseNB * n);
}
inline size_t dense_cnt_offset(int m, int n, int M) {
  return dense_aimg_offset(m, n, M) + align256(sizeof(__half) * static_cast<size_t>(m) * n);
}
inline size_t dense_total(int m, int n, int M) {
  return dense_cnt_offset(m, n, M) +
         align256(sizeof(uint32_t) * static_cast<size_t>(m / kRowBlock) * dense_tiles(M));
}
// K splits of the dense kernel: with fewer units than CTAs, the largest s
// with units * s <= grid, at least 16 stages of 64 columns per split, at most
// 16; else 1.  A split costs its partial sums' L2 reductions and a second
// pass over the block, so it is used only where it fills idle SMs.  (The
// kernel can also split just the last partial round after whole rounds; that
// measured no faster.)
int choose_dense_split(int units, int nstage, int grid);
// K splits of the fused kernel: with fewer units than CTAs, the s (up to 16,
// at least 4 stages per split) that minimises rounds x stages per item plus
// a charge per round for the partial sums of `rows` batch rows; else 1.
int choose_fused_split(int units, int nstage, int grid, int rows);
// Epilogue of the warp-shuffle path: y = binary16(Hb(s_out (.) (scale (.) zacc)))
// per 128-row block (no rotation when s_out is NULL); zeroes zacc.
exl3_status launch_epi(float* zacc, const __half* scales, const __half* s_out, __half* y, int rows,
                       int m, cudaStream_t stream);
exl3_status launch_layer_k1(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k2(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k3(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k4(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k5(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k6(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k7(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_layer_k8(const LayerArgs& a, int mb, cudaStream_t stream);
exl3_status launch_tc_k1(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                          cudaStream_t stream);
exl3_status launch_tc_k2(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                          cudaStream_t stream);
exl3_status launch_tc_k3(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                          cudaStream_t stream);
exl3_status launch_tc_k4(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                          cudaStream_t stream);
exl3_status launch_tc_k5(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                          cudaStream_t stream);
exl3_status launch_tc_k6(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                          cudaStream_t stream);
exl3_status launch_tc_k7(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                          cudaStream_t stream);
exl3_status launch_tc_k8(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                          cudaStream_t stream);

// Kernel parameter blocks of a grouped call stay within the 32764 bytes a
// launch may pass.
static_assert(sizeof(GroupArgs) <= 32764 && sizeof(MvParams) <= 32764 && sizeof(XdupGroup) <= 32764 &&
                  sizeof(EpiGroup) <= 32764 && sizeof(BimgGroup) <= 32764,
              "kernel parameters");

}  // namespace exl3
