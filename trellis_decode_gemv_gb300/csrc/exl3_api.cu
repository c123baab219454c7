// The C ABI of libexl3 (declared in include/exl3.h): host-side validation,
// launch planning and dispatch.  Nothing here allocates, frees or
// synchronizes.
#include <cuda_runtime.h>

#include <atomic>

#include "exl3_host.cuh"

namespace exl3 {

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 1;
  if (dev >= 0 && dev < 64) cache[dev] = sms;
  return sms;
}

LayerPlan plan_layer(int m, int n, int mb, int sm_count) {
  LayerPlan plan;
  const long long tiles = static_cast<long long>(m / 16) * (n / 16);
  const long long per_cta = tiles / sm_count;
  if (mb <= 2 && per_cta < 1024) {
    const long long units = static_cast<long long>(m / kRowBlock) * (n / 16);
    long long ctas = (units + 3) / 4;  // at least 4 tile columns per CTA
    const long long wave = static_cast<long long>(mb == 1 ? 5 : 4) * sm_count;
    if (ctas > wave) ctas = wave;
    plan.ctas = ctas < 1 ? 1 : static_cast<int>(ctas);
    plan.sub = 0;
    return plan;
  }
  const int sub = choose_sub(tiles, mb, sm_count);
  const int nt = n / 16;
  const long long units = static_cast<long long>(m / 16) * ((nt + sub - 1) / sub);
  plan.sub = sub;
  plan.ctas = static_cast<int>(units < sm_count ? units : sm_count);
  return plan;
}

int choose_sub(long long tiles, int mb, int sm_count) {
  const int warps = mb <= 2 ? 32 : mb == 4 ? 16 : 8;
  const long long per_cta = tiles / sm_count;
  // (per-sub-unit work -- the layer lookup, the row index, the reduction --
  // is a few per cent of a 16-tile sub-unit's instructions at batch 1)
  if (mb == 1 && per_cta >= 32LL * 2 * warps) return 32;
  if (per_cta >= 16LL * 2 * warps) return 16;
  if (per_cta >= 8LL * 2 * warps) return 8;
  return 4;
}

namespace {

std::atomic<int> g_path{EXL3_PATH_AUTO};
std::atomic<int> g_prefill{EXL3_PREFILL_AUTO};
std::atomic<int> g_debug_stall{0};

exl3_status launch_tc(const LayerArgs& a, const __half* bimg, const float* bsum, int M, int grid,
                      cudaStream_t stream) {
  switch (a.K) {
    case 1: return launch_tc_k1(a, bimg, bsum, M, grid, stream);
    case 2: return launch_tc_k2(a, bimg, bsum, M, grid, stream);
    case 3: return launch_tc_k3(a, bimg, bsum, M, grid, stream);
    case 4: return launch_tc_k4(a, bimg, bsum, M, grid, stream);
    case 5: return launch_tc_k5(a, bimg, bsum, M, grid, stream);
    case 6: return launch_tc_k6(a, bimg, bsum, M, grid, stream);
    case 7: return launch_tc_k7(a, bimg, bsum, M, grid, stream);
    case 8: return launch_tc_k8(a, bimg, bsum, M, grid, stream);
    default: return EXL3_ERR_K;
  }
}

exl3_status launch_group_kset(const GroupArgs& a, int K, cudaStream_t stream) {
  switch (K) {
    case 1: return launch_group_kset_k1(a, stream);
    case 2: return launch_group_kset_k2(a, stream);
    case 3: return launch_group_kset_k3(a, stream);
    case 4: return launch_group_kset_k4(a, stream);
    case 5: return launch_group_kset_k5(a, stream);
    case 6: return launch_group_kset_k6(a, stream);
    case 7: return launch_group_kset_k7(a, stream);
    case 8: return launch_group_kset_k8(a, stream);
    default: return EXL3_ERR_K;
  }
}

exl3_status launch_group(const GroupArgs& a, int K, int codebook, int mb, cudaStream_t stream) {
  switch (K) {
    case 1: return launch_group_k1(a, codebook, mb, stream);
    case 2: return launch_group_k2(a, codebook, mb, stream);
    case 3: return launch_group_k3(a, codebook, mb, stream);
    case 4: return launch_group_k4(a, codebook, mb, stream);
    case 5: return launch_group_k5(a, codebook, mb, stream);
    case 6: return launch_group_k6(a, codebook, mb, stream);
    case 7: return launch_group_k7(a, codebook, mb, stream);
    case 8: return launch_group_k8(a, codebook, mb, stream);
    default: return EXL3_ERR_K;
  }
}

exl3_status launch_layer(const LayerArgs& a, int mb, cudaStream_t stream) {
  switch (a.K) {
    case 1: return launch_layer_k1(a, mb, stream);
    case 2: return launch_layer_k2(a, mb, stream);
    case 3: return launch_layer_k3(a, mb, stream);
    case 4: return launch_layer_k4(a, mb, stream);
    case 5: return launch_layer_k5(a, mb, stream);
    case 6: return launch_layer_k6(a, mb, stream);
    case 7: return launch_layer_k7(a, mb, stream);
    case 8: return launch_layer_k8(a, mb, stream);
    default: return EXL3_ERR_K;
  }
}

exl3_status launch_mv(const MvParams& p, int K, int codebook, int grid, cudaStream_t stream) {
  switch (K) {
    case 1: return launch_mv_k1(p, codebook, grid, stream);
    case 2: return launch_mv_k2(p, codebook, grid, stream);
    case 3: return launch_mv_k3(p, codebook, grid, stream);
    case 4: return launch_mv_k4(p, codebook, grid, stream);
    case 5: return launch_mv_k5(p, codebook, grid, stream);
    case 6: return launch_mv_k6(p, codebook, grid, stream);
    case 7: return launch_mv_k7(p, codebook, grid, stream);
    case 8: return launch_mv_k8(p, codebook, grid, stream);
    default: return EXL3_ERR_K;
  }
}

int batch_chunk(int rem) { return rem >= 8 ? 8 : rem >= 4 ? 4 : rem >= 2 ? 2 : 1; }

// Kernel family of a call of M <= EXL3_MAX_BATCH rows: the warp-shuffle
// kernels at M <= 2 (and whenever exl3_set_path selects them), the
// decode-MMA kernel above (and whenever EXL3_PATH_TENSOR selects it).  At
// batch 1 the warp-shuffle kernels decode and multiply in the same 32 warps
// per SM; the decode-MMA kernel's decoders, issuers and epilogue warps spend
// too much of each chunk on their hand-offs to beat them there (measured).
bool use_shuffle(int M) {
  const int path = g_path.load(std::memory_order_relaxed);
  return path == EXL3_PATH_SHUFFLE || (path == EXL3_PATH_AUTO && M <= 2);
}

// Prefill strategy above EXL3_MAX_BATCH rows (outside EXL3_PATH_TENSOR): the
// fused kernel decodes every tile once per batch tile, the decode-once path
// once per call plus a round trip of the decoded matrix through HBM.
constexpr int kFusedMaxRows = 256;
bool prefill_fused(int M) {
  const int s = g_prefill.load(std::memory_order_relaxed);
  return s == EXL3_PREFILL_FUSED || (s == EXL3_PREFILL_AUTO && M <= kFusedMaxRows);
}
// Batch tile of the fused kernel: one tile of 64 rows up to 64, of 128 up to
// 128, else tiles of 256.
int fused_nb(int M) { return M <= 64 ? 64 : M <= 128 ? 128 : 256; }

}  // namespace

exl3_status run_tensor(LayerArgs a, int M, float* zacc, uint32_t* status, __half* bimg, float* bsum,
                       cudaStream_t cs) {
  // x-tilde as operand-B images (and, for 1MAD, its block sums), then the
  // persistent tensor-core kernel into zacc, then the output transform; the
  // last two are programmatic dependents of the kernel before them.
  a.zacc = zacc;
  a.status = status;
  if (a.codebook != EXL3_CB_1MAD && a.codebook != EXL3_CB_MUL1) bsum = nullptr;
  exl3_status st = launch_bimg(a.x, a.s_in, bimg, bsum, M, kPrefillRows, a.n, cs);
  if (st != EXL3_OK) return st;
  if ((st = launch_tc(a, bimg, bsum, M, device_sm_count(), cs)) != EXL3_OK) return st;
  return launch_epi(a.zacc, a.scales, a.s_out, a.y, M, a.m, cs);
}

// The decode-MMA kernel loads the codes of a chunk (eight tile-row strips of
// 8 tiles) with one 2-D tensor copy: the codes as (m/16) rows of (n/16) * 4K
// 64-bit elements, a box of 32K x 8.
// The driver's tensor-map encoder, looked up through the runtime (so that the
// library loads, for its host-side checks, where no driver is installed).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
      return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

exl3_status mv_codes_map(CUtensorMap* map, const uint32_t* codes, int K, int m, int n) {
  const EncodeTiledFn encode = encode_tiled();
  if (encode == nullptr) return EXL3_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(n / 16) * 4 * K, static_cast<cuuint64_t>(m / 16)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(n / 16) * 8 * K * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(32 * K), 8u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint32_t*>(codes), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? EXL3_OK : EXL3_ERR_CUDA;
}

exl3_status run_mv(MvParams p, int K, int codebook, cudaStream_t cs) {
  int units = 0;
  exl3_status st;
  for (int i = 0; i < p.count; ++i) {
    if ((st = mv_codes_map(&p.l[i].codes_map, p.l[i].codes, K, p.l[i].m, p.l[i].n)) != EXL3_OK) return st;
    p.l[i].nkb = p.l[i].n / kMvChunkCols;
    p.l[i].u_begin = units;
    units += (p.l[i].m / kRowBlock) * p.l[i].nkb;
  }
  p.units = units;
  const int sms = device_sm_count();
  const int grid = units < sms ? units : sms;
  if (p.M > 2) {
    // one operand-image launch for every layer of the call
    BimgGroup bg{};
    bg.count = p.count;
    for (int i = 0; i < p.count; ++i)
      bg.e[i] = BimgEntry{p.l[i].x, p.l[i].s_in, const_cast<__half*>(p.l[i].bimg),
                          mv_centred(codebook) ? const_cast<float*>(p.l[i].bsum) : nullptr, p.l[i].n, 0};
    if ((st = launch_bimg_group(bg, p.M, mv_nb(p.M), cs)) != EXL3_OK) return st;
  }
  return launch_mv(p, K, codebook, grid, cs);
}

exl3_status run_shuffle(LayerArgs a, int M, float* zacc, uint32_t* xd, cudaStream_t cs) {
  const int sms = device_sm_count();
  a.zacc = zacc;
  const __half* x = a.x;
  __half* y = a.y;
  exl3_status st;
  for (int done = 0; done < M;) {
    const int mb = batch_chunk(M - done);
    a.x = x + static_cast<size_t>(done) * a.n;
    a.y = y + static_cast<size_t>(done) * a.m;
    const LayerPlan plan = plan_layer(a.m, a.n, mb, sms);
    if (plan.sub == 0) {
      a.ctas = plan.ctas;
      if ((st = launch_layer(a, mb, cs)) != EXL3_OK) return st;
    } else {
      if ((st = launch_xdup(a.x, a.s_in, xd, mb, a.n, a.codebook, cs)) != EXL3_OK) return st;
      GroupArgs g{};
      g.count = 1;
      g.sub = plan.sub;
      g.l[0].codes = a.codes;
      g.l[0].xdup = xd;
      g.l[0].zacc = zacc;
      g.l[0].m = a.m;
      g.l[0].n = a.n;
      g.l[0].u_begin = 0;
      g.l[0].per_row = (a.n / 16 + plan.sub - 1) / plan.sub;
      g.units = (a.m / 16) * g.l[0].per_row;
      g.l[0].row_magic = div_magic(g.l[0].per_row, g.units);
      g.ctas = plan.ctas;
      if ((st = launch_group(g, a.K, a.codebook, mb, cs)) != EXL3_OK) return st;
    }
    if ((st = launch_epi(zacc, a.scales, a.s_out, a.y, mb, a.m, cs)) != EXL3_OK) return st;
    done += mb;
  }
  return EXL3_OK;
}

}  // namespace exl3

using namespace exl3;

extern "C" const char* exl3_status_string(exl3_status status) {
  switch (status) {
    case EXL3_OK: return "ok";
    case EXL3_ERR_NULL: return "a required pointer is NULL";
    case EXL3_ERR_SHAPE: return "m and n must be positive multiples of 128 (and n within the supported maximum)";
    case EXL3_ERR_K: return "K (bits per weight) must be in 1..8";
    case EXL3_ERR_CODEBOOK: return "unknown codebook id (0 = 3INST, 1 = 1MAD)";
    case EXL3_ERR_BATCH: return "batch M out of range";
    case EXL3_ERR_ALIGN: return "device pointers must be 16-byte aligned";
    case EXL3_ERR_WORKSPACE: return "workspace missing or smaller than exl3_workspace_bytes()";
    case EXL3_ERR_CUDA: return "CUDA launch error";
    case EXL3_ERR_DEVICE_CHECK: return "device-side check failed";
    case EXL3_ERR_SCRATCH: return "layer needs more scratch than exl3_gemv_noalloc's fixed array (EXL3_NOALLOC_SCRATCH_BYTES)";
  }
  return "unknown status";
}

extern "C" const char* exl3_version(void) { return "libexl3 0.2.0 sm_103a"; }

extern "C" exl3_status exl3_set_prefill(int strategy) {
  if (strategy != EXL3_PREFILL_AUTO && strategy != EXL3_PREFILL_FUSED && strategy != EXL3_PREFILL_DECODE_ONCE)
    return EXL3_ERR_BATCH;
  g_prefill.store(strategy, std::memory_order_relaxed);
  return EXL3_OK;
}

extern "C" exl3_status exl3_set_path(int path) {
  if (path != EXL3_PATH_AUTO && path != EXL3_PATH_SHUFFLE && path != EXL3_PATH_TENSOR)
    return EXL3_ERR_BATCH;
  g_path.store(path, std::memory_order_relaxed);
  return EXL3_OK;
}

extern "C" exl3_status exl3_device_status(const void* status_word, exl3_stream_t stream) {
  if (status_word == nullptr) return EXL3_ERR_NULL;
  uint32_t word = 0;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, status_word, sizeof(word), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
    return EXL3_ERR_CUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return EXL3_ERR_CUDA;
  return word == 0u ? EXL3_OK : EXL3_ERR_DEVICE_CHECK;
}

extern "C" exl3_status exl3_debug_stall_tensor_wait(int on) {
  g_debug_stall.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
  return EXL3_OK;
}

extern "C" size_t exl3_workspace_bytes(int m, int n, int M) {
  if (check_shape(m, n) != EXL3_OK || M < 1 || M > EXL3_MAX_BATCH) return 0;
  return workspace_total(m, n, M);
}

extern "C" exl3_status exl3_rht_in(const exl3_half* x, const exl3_half* s_in, exl3_half* x_rot,
                                   int M, int n, exl3_stream_t stream) {
  if (M < 1) return EXL3_ERR_BATCH;
  if (n <= 0 || n % kRowBlock) return EXL3_ERR_SHAPE;
  if (!x || !s_in || !x_rot) return EXL3_ERR_NULL;
  if (!aligned16(x) || !aligned16(s_in) || !aligned16(x_rot)) return EXL3_ERR_ALIGN;
  return launch_rht(reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(s_in),
                    reinterpret_cast<__half*>(x_rot), M, n, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" exl3_status exl3_rht_out(const exl3_half* z, const exl3_half* s_out, exl3_half* y,
                                    int M, int m, exl3_stream_t stream) {
  return exl3_rht_in(z, s_out, y, M, m, stream);
}

extern "C" exl3_status exl3_decode_tiles(const uint32_t* codes, int K, int codebook, int m, int n,
                                         exl3_half* w_out, exl3_stream_t stream) {
  exl3_status st = check_shape(m, n);
  if (st != EXL3_OK) return st;
  if ((st = check_k_cb(K, codebook)) != EXL3_OK) return st;
  if (!codes || !w_out) return EXL3_ERR_NULL;
  if (!aligned16(codes) || !aligned16(w_out)) return EXL3_ERR_ALIGN;
  return launch_decode(codes, K, codebook, m, n, reinterpret_cast<__half*>(w_out),
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" exl3_status exl3_gemm_small(const uint32_t* codes, int K, int codebook, int m, int n,
                                       const exl3_half* s_in, const exl3_half* s_out,
                                       const exl3_half* scales, int M, const exl3_half* x,
                                       exl3_half* y, void* workspace, size_t workspace_bytes,
                                       exl3_stream_t stream) {
  exl3_status st = check_shape(m, n);
  if (st != EXL3_OK) return st;
  if ((st = check_k_cb(K, codebook)) != EXL3_OK) return st;
  if (M < 1 || M > EXL3_MAX_BATCH) return EXL3_ERR_BATCH;
  if (!codes || !scales || !x || !y) return EXL3_ERR_NULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(y) ||
      (s_in && !aligned16(s_in)) || (s_out && !aligned16(s_out)))
    return EXL3_ERR_ALIGN;
  const size_t need = exl3_workspace_bytes(m, n, M);
  if (!workspace || workspace_bytes < need) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;

  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  LayerArgs a{};
  a.codes = codes;
  a.K = K;
  a.codebook = codebook;
  a.m = m;
  a.n = n;
  a.s_in = reinterpret_cast<const __half*>(s_in);
  a.s_out = reinterpret_cast<const __half*>(s_out);
  a.scales = reinterpret_cast<const __half*>(scales);
  a.x = reinterpret_cast<const __half*>(x);
  a.y = reinterpret_cast<__half*>(y);
  a.debug_stall = g_debug_stall.load(std::memory_order_relaxed);
  char* ws = static_cast<char*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws) + m / kRowBlock;
  float* zacc = reinterpret_cast<float*>(ws + zacc_offset(m));
  if (!use_shuffle(M)) {
    MvParams p{};
    p.count = 1;
    p.M = M;
    p.status = status;
    p.debug_stall = a.debug_stall;
    MvLayer& L = p.l[0];
    L.codes = codes;
    L.x = a.x;
    L.s_in = a.s_in;
    L.bimg = reinterpret_cast<const __half*>(ws + bimg_offset(m, M));
    L.bsum = reinterpret_cast<const float*>(ws + bsum_offset(m, n, M));
    L.scales = a.scales;
    L.s_out = a.s_out;
    L.y = a.y;
    L.zacc = zacc;
    L.cnt = reinterpret_cast<uint32_t*>(ws);
    L.m = m;
    L.n = n;
    return run_mv(p, K, codebook, cs);
  }
  // x pairs of each batch chunk go where the tensor path keeps its operand
  // images (at least 32 n bytes, enough for 8 rows of n 32-bit pairs).
  return run_shuffle(a, M, zacc, reinterpret_cast<uint32_t*>(ws + bimg_offset(m, M)), cs);
}

namespace {

// Workspace of a group: the status word (first 256 bytes), then per layer its
// block counters (m/128 words) and fp32 row sums [M][m], both zero on entry
// and exit, then per layer one scratch region: the x pairs of the warp-shuffle
// path ([min(M, 8)][n] words) or the decode-MMA kernel's operand images.
struct GroupLayout {
  size_t cnt[kMaxGroup], zacc[kMaxGroup], scratch[kMaxGroup];
  size_t total;
};

GroupLayout group_layout(const exl3_layer* L, int count, int M) {
  GroupLayout g{};
  const size_t mb = static_cast<size_t>(M < 8 ? M : 8);
  size_t off = 256;
  for (int i = 0; i < count; ++i) {
    g.cnt[i] = off;
    off += align256(sizeof(uint32_t) * (L[i].m / kRowBlock));
    g.zacc[i] = off;
    off += align256(sizeof(float) * static_cast<size_t>(M) * L[i].m);
  }
  for (int i = 0; i < count; ++i) {
    g.scratch[i] = off;
    const size_t xd = sizeof(uint32_t) * mb * L[i].n;
    const size_t img = M > 2 ? align256(mv_bimg_bytes(L[i].n, M)) + mv_bsum_bytes(L[i].n, M) : 0;
    off += align256(xd > img ? xd : img);
  }
  g.total = off;
  return g;
}

}  // namespace

extern "C" size_t exl3_group_workspace_bytes(const exl3_layer* layers, int count, int M) {
  if (layers == nullptr || count < 1 || count > EXL3_MAX_GROUP || M < 1 || M > EXL3_MAX_BATCH) return 0;
  for (int i = 0; i < count; ++i)
    if (check_shape(layers[i].m, layers[i].n) != EXL3_OK) return 0;
  return group_layout(layers, count, M).total;
}

namespace {

exl3_status check_group_layers(const exl3_layer* layers, int count) {
  exl3_status st;
  for (int i = 0; i < count; ++i) {
    const exl3_layer& L = layers[i];
    if ((st = check_shape(L.m, L.n)) != EXL3_OK) return st;
    if (!L.codes || !L.scales || !L.x || !L.y) return EXL3_ERR_NULL;
    if (!aligned16(L.codes) || !aligned16(L.scales) || !aligned16(L.x) || !aligned16(L.y) ||
        (L.s_in && !aligned16(L.s_in)) || (L.s_out && !aligned16(L.s_out)))
      return EXL3_ERR_ALIGN;
  }
  return EXL3_OK;
}

// The layers idx[0 .. count) of `layers`, each of its own K (ks[j]) and code
// (codes[j]), with the per-layer workspace regions of gl.  Warp-shuffle path:
// per batch chunk one kernel chain -- the x pairs of every layer, then one
// sub-unit kernel per (K, code) class over the tiles of that class's layers
// (the classes in order of first appearance, each a programmatic dependent of
// the one before), then the output transform of every layer.  Decode-MMA
// path: one call of it per class.
exl3_status group_chain(const exl3_layer* layers, const int* idx, int count, const int* ks, const int* codes, int M,
                        const GroupLayout& gl, char* ws, cudaStream_t cs) {
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  exl3_status st;
  // the classes: cls[j] = index of layer j's (K, code) among the distinct pairs
  int cls[kMaxGroup], ncls = 0, cls_k[kMaxGroup], cls_cb[kMaxGroup];
  for (int j = 0; j < count; ++j) {
    int c = 0;
    while (c < ncls && !(cls_k[c] == ks[j] && cls_cb[c] == codes[j])) ++c;
    if (c == ncls) {
      cls_k[c] = ks[j];
      cls_cb[c] = codes[j];
      ++ncls;
    }
    cls[j] = c;
  }
  if (!use_shuffle(M)) {
    for (int c = 0; c < ncls; ++c) {
      const int K = cls_k[c], codebook = cls_cb[c];
      MvParams p{};
      p.M = M;
      p.status = status;
      p.debug_stall = g_debug_stall.load(std::memory_order_relaxed);
      for (int j = 0; j < count; ++j) {
        if (cls[j] != c) continue;
        const int i = idx[j];
        const exl3_layer& L = layers[i];
        MvLayer& d = p.l[p.count++];
        d.codes = L.codes;
        d.x = reinterpret_cast<const __half*>(L.x);
        d.s_in = reinterpret_cast<const __half*>(L.s_in);
        d.bimg = reinterpret_cast<const __half*>(ws + gl.scratch[i]);
        d.bsum = reinterpret_cast<const float*>(ws + gl.scratch[i] + align256(mv_bimg_bytes(L.n, M)));
        d.scales = reinterpret_cast<const __half*>(L.scales);
        d.s_out = reinterpret_cast<const __half*>(L.s_out);
        d.y = reinterpret_cast<__half*>(L.y);
        d.zacc = reinterpret_cast<float*>(ws + gl.zacc[i]);
        d.cnt = reinterpret_cast<uint32_t*>(ws + gl.cnt[i]);
        d.m = L.m;
        d.n = L.n;
      }
      if ((st = run_mv(p, K, codebook, cs)) != EXL3_OK) return st;
    }
    return EXL3_OK;
  }

  // Warp-shuffle path.
  const int sms = device_sm_count();
  long long tiles[kMaxGroup] = {};  // per class
  for (int j = 0; j < count; ++j)
    tiles[cls[j]] += static_cast<long long>(layers[idx[j]].m / 16) * (layers[idx[j]].n / 16);
  for (int done = 0; done < M;) {
    const int mb = batch_chunk(M - done);
    XdupGroup xg{};
    EpiGroup eg{};
    xg.count = eg.count = count;
    xg.rows = eg.rows = mb;
    for (int j = 0; j < count; ++j) {
      const int i = idx[j];
      const exl3_layer& L = layers[i];
      float* zacc = reinterpret_cast<float*>(ws + gl.zacc[i]);
      uint32_t* xd = reinterpret_cast<uint32_t*>(ws + gl.scratch[i]);
      xg.e[j].x = reinterpret_cast<const __half*>(L.x) + static_cast<size_t>(done) * L.n;
      xg.e[j].s_in = reinterpret_cast<const __half*>(L.s_in);
      xg.e[j].xd = xd;
      xg.e[j].n = L.n;
      xg.e[j].factor = code_x_factor(codes[j]);
      eg.e[j].zacc = zacc;
      eg.e[j].scales = reinterpret_cast<const __half*>(L.scales);
      eg.e[j].s_out = reinterpret_cast<const __half*>(L.s_out);
      eg.e[j].y = reinterpret_cast<__half*>(L.y) + static_cast<size_t>(done) * L.m;
      eg.e[j].m = L.m;
    }
    if ((st = launch_xdup_group(xg, -1, cs)) != EXL3_OK) return st;
    bool launched[kMaxGroup] = {};
    for (int c = 0; c < ncls; ++c) {
      if (launched[c]) continue;
      if (mb == 1) {
        // the classes of this K: at 32-tile sub-units, one launch for all of them
        const int K = cls_k[c];
        long long ktiles = 0;
        int nk = 0;
        for (int c2 = c; c2 < ncls; ++c2)
          if (cls_k[c2] == K) {
            ktiles += tiles[c2];
            ++nk;
          }
        if (nk > 1 && choose_sub(ktiles, 1, sms) == 32) {
          GroupArgs g{};
          g.sub = 32;
          int units = 0;
          for (int code = 0; code < 4; ++code) {
            for (int j = 0; j < count; ++j) {
              if (ks[j] != K || codes[j] != code) continue;
              const int i = idx[j];
              const exl3_layer& L = layers[i];
              GroupLayer& d = g.l[g.count++];
              d.codes = L.codes;
              d.xdup = reinterpret_cast<uint32_t*>(ws + gl.scratch[i]);
              d.zacc = reinterpret_cast<float*>(ws + gl.zacc[i]);
              d.m = L.m;
              d.n = L.n;
              d.u_begin = units;
              d.per_row = (L.n / 16 + 31) / 32;
              d.row_magic = div_magic(d.per_row, static_cast<long long>(L.m / 16) * d.per_row);
              units += (L.m / 16) * d.per_row;
            }
            g.code_end[code] = units;
          }
          g.units = units;
          g.ctas = units < sms ? units : sms;
          if ((st = launch_group_kset(g, K, cs)) != EXL3_OK) return st;
          for (int c2 = c; c2 < ncls; ++c2)
            if (cls_k[c2] == K) launched[c2] = true;
          continue;
        }
      }
      GroupArgs g{};
      const int sub = choose_sub(tiles[c], mb, sms);
      g.sub = sub;
      int units = 0;
      for (int j = 0; j < count; ++j) {
        if (cls[j] != c) continue;
        const int i = idx[j];
        const exl3_layer& L = layers[i];
        GroupLayer& d = g.l[g.count++];
        d.codes = L.codes;
        d.xdup = reinterpret_cast<uint32_t*>(ws + gl.scratch[i]);
        d.zacc = reinterpret_cast<float*>(ws + gl.zacc[i]);
        d.m = L.m;
        d.n = L.n;
        d.u_begin = units;
        d.per_row = (L.n / 16 + sub - 1) / sub;
        d.row_magic = div_magic(d.per_row, static_cast<long long>(L.m / 16) * d.per_row);
        units += (L.m / 16) * d.per_row;
      }
      g.units = units;
      g.ctas = units < sms ? units : sms;
      if ((st = launch_group(g, cls_k[c], cls_cb[c], mb, cs)) != EXL3_OK) return st;
    }
    if ((st = launch_epi_group(eg, cs)) != EXL3_OK) return st;
    done += mb;
  }
  return EXL3_OK;
}

}  // namespace

extern "C" exl3_status exl3_gemm_grouped(const exl3_layer* layers, int count, int K, int codebook, int M,
                                         void* workspace, size_t workspace_bytes, exl3_stream_t stream) {
  if (layers == nullptr) return EXL3_ERR_NULL;
  if (count < 1 || count > EXL3_MAX_GROUP) return EXL3_ERR_BATCH;
  exl3_status st = check_k_cb(K, codebook);
  if (st != EXL3_OK) return st;
  if (M < 1 || M > EXL3_MAX_BATCH) return EXL3_ERR_BATCH;
  if ((st = check_group_layers(layers, count)) != EXL3_OK) return st;
  const size_t need = exl3_group_workspace_bytes(layers, count, M);
  if (!workspace || workspace_bytes < need) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;

  const GroupLayout gl = group_layout(layers, count, M);
  int idx[kMaxGroup], ks[kMaxGroup], codes[kMaxGroup];
  for (int i = 0; i < count; ++i) {
    idx[i] = i;
    ks[i] = K;
    codes[i] = codebook;
  }
  return group_chain(layers, idx, count, ks, codes, M, gl, static_cast<char*>(workspace),
                     reinterpret_cast<cudaStream_t>(stream));
}

namespace {

// The plain layers of a multi-code group (their shapes set the workspace).
void plain_layers(const exl3_layer_kc* layers, int count, exl3_layer* out) {
  for (int i = 0; i < count; ++i) out[i] = layers[i].layer;
}

}  // namespace

extern "C" size_t exl3_multi_workspace_bytes(const exl3_layer_kc* layers, int count, int M) {
  if (layers == nullptr || count < 1 || count > EXL3_MAX_GROUP) return 0;
  exl3_layer plain[kMaxGroup];
  plain_layers(layers, count, plain);
  return exl3_group_workspace_bytes(plain, count, M);
}

extern "C" exl3_status exl3_gemm_multi(const exl3_layer_kc* layers, int count, int M, void* workspace,
                                       size_t workspace_bytes, exl3_stream_t stream) {
  if (layers == nullptr) return EXL3_ERR_NULL;
  if (count < 1 || count > EXL3_MAX_GROUP) return EXL3_ERR_BATCH;
  if (M < 1 || M > EXL3_MAX_BATCH) return EXL3_ERR_BATCH;
  exl3_status st;
  for (int i = 0; i < count; ++i)
    if ((st = check_k_cb(layers[i].K, layers[i].codebook)) != EXL3_OK) return st;
  exl3_layer plain[kMaxGroup];
  plain_layers(layers, count, plain);
  if ((st = check_group_layers(plain, count)) != EXL3_OK) return st;
  const size_t need = exl3_group_workspace_bytes(plain, count, M);
  if (!workspace || workspace_bytes < need) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;

  const GroupLayout gl = group_layout(plain, count, M);
  int idx[kMaxGroup], ks[kMaxGroup], codes[kMaxGroup];
  for (int i = 0; i < count; ++i) {
    idx[i] = i;
    ks[i] = layers[i].K;
    codes[i] = layers[i].codebook;
  }
  return group_chain(plain, idx, count, ks, codes, M, gl, static_cast<char*>(workspace),
                     reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t exl3_gemm_workspace_bytes(int m, int n, int M) {
  if (check_shape(m, n) != EXL3_OK || M < 1) return 0;
  if (M <= EXL3_MAX_BATCH) return exl3_workspace_bytes(m, n, M);
  // Either prefill strategy may run (exl3_set_path can change between calls).
  const size_t dense = dense_total(m, n, M);
  const size_t passes = workspace_total(m, n, kPrefillRows);
  return dense > passes ? dense : passes;
}

extern "C" int exl3_gemm_launches(int m, int n, int M) {
  if (check_shape(m, n) != EXL3_OK || M < 1) return 0;
  const int path = g_path.load(std::memory_order_relaxed);
  if (M <= EXL3_MAX_BATCH) {
    if (!use_shuffle(M)) return mv_launches(1, M);
    // warp-shuffle path: per batch chunk the layer kernel (plus the x-pair
    // kernel in front of the sub-unit kernel) and the output kernel
    const int sms = device_sm_count();
    int launches = 0;
    for (int done = 0; done < M;) {
      const int mb = batch_chunk(M - done);
      launches += plan_layer(m, n, mb, sms).sub == 0 ? 2 : 3;
      done += mb;
    }
    return launches;
  }
  if (path == EXL3_PATH_TENSOR) return 3 * ((M + kPrefillRows - 1) / kPrefillRows);
  return prefill_fused(M) ? 2 : 3;
}

namespace {

// Fused prefill: x-tilde into operand-B images, then the dense kernel that
// decodes its operand A from the codes in shared memory.
exl3_status run_fused(const LayerArgs& a, int M, char* ws, cudaStream_t cs) {
  uint32_t* status = reinterpret_cast<uint32_t*>(ws) + a.m / kRowBlock;
  float* zacc = reinterpret_cast<float*>(ws + zacc_offset(a.m));
  __half* bimg = reinterpret_cast<__half*>(ws + dense_bimg_offset(a.m, M));
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + dense_cnt_offset(a.m, a.n, M));
  const int nb = fused_nb(M);
  exl3_status st = launch_bimg(a.x, a.s_in, bimg, nullptr, M, nb, a.n, cs);
  if (st != EXL3_OK) return st;
  const int units = (a.m / kRowBlock) * ((M + nb - 1) / nb);
  const int split = choose_fused_split(units, a.n / 64, device_sm_count(), M < nb ? M : nb);
  return launch_fused(a.codes, a.K, a.codebook, bimg, a.scales, a.s_out, a.y, zacc, cnt, a.m, a.n, M, nb, split,
                      status, a.debug_stall, cs);
}

// Decode once, dense GEMM: W-hat into operand-A images, x-tilde into
// operand-B images, then the dense kernel.
exl3_status run_dense(const LayerArgs& a, int M, char* ws, cudaStream_t cs) {
  uint32_t* status = reinterpret_cast<uint32_t*>(ws) + a.m / kRowBlock;
  float* zacc = reinterpret_cast<float*>(ws + zacc_offset(a.m));
  __half* bimg = reinterpret_cast<__half*>(ws + dense_bimg_offset(a.m, M));
  unsigned char* aimg = reinterpret_cast<unsigned char*>(ws + dense_aimg_offset(a.m, a.n, M));
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + dense_cnt_offset(a.m, a.n, M));
  exl3_status st = launch_decode_aimg(a.codes, a.K, a.codebook, a.m, a.n, aimg, cs);
  if (st != EXL3_OK) return st;
  const int nb = dense_nb(M);
  if ((st = launch_bimg(a.x, a.s_in, bimg, nullptr, M, nb, a.n, cs)) != EXL3_OK) return st;
  const int units = (a.m / kRowBlock) * ((M + nb - 1) / nb);
  const int split = choose_dense_split(units, a.n / 64, device_sm_count());
  return launch_dense(aimg, bimg, a.scales, a.s_out, a.y, zacc, cnt, a.m, a.n, M, nb, split, status,
                      a.debug_stall, cs);
}

}  // namespace

extern "C" exl3_status exl3_gemm(const uint32_t* codes, int K, int codebook, int m, int n,
                                 const exl3_half* s_in, const exl3_half* s_out,
                                 const exl3_half* scales, int M, const exl3_half* x, exl3_half* y,
                                 void* workspace, size_t workspace_bytes, exl3_stream_t stream) {
  if (M < 1) return EXL3_ERR_BATCH;
  if (M <= EXL3_MAX_BATCH)
    return exl3_gemm_small(codes, K, codebook, m, n, s_in, s_out, scales, M, x, y, workspace,
                           workspace_bytes, stream);
  exl3_status st = check_shape(m, n);
  if (st != EXL3_OK) return st;
  if ((st = check_k_cb(K, codebook)) != EXL3_OK) return st;
  if (!codes || !scales || !x || !y) return EXL3_ERR_NULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(y) ||
      (s_in && !aligned16(s_in)) || (s_out && !aligned16(s_out)))
    return EXL3_ERR_ALIGN;
  if (!workspace || workspace_bytes < exl3_gemm_workspace_bytes(m, n, M)) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if (g_path.load(std::memory_order_relaxed) != EXL3_PATH_TENSOR) {
    LayerArgs a{};
    a.codes = codes;
    a.K = K;
    a.codebook = codebook;
    a.m = m;
    a.n = n;
    a.s_in = reinterpret_cast<const __half*>(s_in);
    a.s_out = reinterpret_cast<const __half*>(s_out);
    a.scales = reinterpret_cast<const __half*>(scales);
    a.x = reinterpret_cast<const __half*>(x);
    a.y = reinterpret_cast<__half*>(y);
    a.debug_stall = g_debug_stall.load(std::memory_order_relaxed);
    return prefill_fused(M) ? run_fused(a, M, ws, cs) : run_dense(a, M, ws, cs);
  }
  // EXL3_PATH_TENSOR: passes of up to 128 batch rows through the tensor-core
  // kernel at N = 128; each pass decodes the tiles once into tensor memory for
  // all its rows.
  const int R = kPrefillRows;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws) + m / kRowBlock;
  float* zacc = reinterpret_cast<float*>(ws + zacc_offset(m));
  __half* bimg = reinterpret_cast<__half*>(ws + bimg_offset(m, R));
  float* bsum = reinterpret_cast<float*>(ws + bsum_offset(m, n, R));
  for (int done = 0; done < M; done += R) {
    const int rows = M - done < R ? M - done : R;
    LayerArgs a{};
    a.codes = codes;
    a.K = K;
    a.codebook = codebook;
    a.m = m;
    a.n = n;
    a.s_in = reinterpret_cast<const __half*>(s_in);
    a.s_out = reinterpret_cast<const __half*>(s_out);
    a.scales = reinterpret_cast<const __half*>(scales);
    a.x = reinterpret_cast<const __half*>(x) + static_cast<size_t>(done) * n;
    a.y = reinterpret_cast<__half*>(y) + static_cast<size_t>(done) * m;
    a.debug_stall = g_debug_stall.load(std::memory_order_relaxed);
    // a last pass of fewer rows runs the same N = 128 kernel (rows past it zero)
    if ((st = run_tensor(a, rows, zacc, status, bimg, bsum, cs)) != EXL3_OK) return st;
  }
  return EXL3_OK;
}

extern "C" exl3_status exl3_gemv(const uint32_t* codes, int K, int codebook, int m, int n,
                                 const exl3_half* s_in, const exl3_half* s_out,
                                 const exl3_half* scales, const exl3_half* x, exl3_half* y,
                                 void* workspace, size_t workspace_bytes, exl3_stream_t stream) {
  return exl3_gemm_small(codes, K, codebook, m, n, s_in, s_out, scales, 1, x, y, workspace,
                         workspace_bytes, stream);
}
