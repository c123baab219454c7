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
  const int warps = mb == 1 ? 32 : mb == 2 ? 24 : mb == 4 ? 16 : 8;
  int sub = 4;
  if (per_cta >= 16LL * 2 * warps) {
    sub = 16;
  } else if (per_cta >= 8LL * 2 * warps) {
    sub = 8;
  }
  const int nt = n / 16;
  const long long units = static_cast<long long>(m / 16) * ((nt + sub - 1) / sub);
  plan.sub = sub;
  plan.ctas = static_cast<int>(units < sm_count ? units : sm_count);
  return plan;
}

namespace {

std::atomic<int> g_path{EXL3_PATH_AUTO};
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

}  // namespace
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

extern "C" exl3_status exl3_set_path(int path) {
  if (path != EXL3_PATH_AUTO && path != EXL3_PATH_SHUFFLE && path != EXL3_PATH_TENSOR)
    return EXL3_ERR_BATCH;
  g_path.store(path, std::memory_order_relaxed);
  return EXL3_OK;
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
  const int sms = device_sm_count();
  LayerArgs a{};
  a.codes = codes;
  a.K = K;
  a.codebook = codebook;
  a.m = m;
  a.n = n;
  a.s_in = reinterpret_cast<const __half*>(s_in);
  a.s_out = reinterpret_cast<const __half*>(s_out);
  a.scales = reinterpret_cast<const __half*>(scales);
  char* ws = static_cast<char*>(workspace);
  a.counters = reinterpret_cast<uint32_t*>(ws);
  a.status = a.counters + m / kRowBlock;
  a.zacc = reinterpret_cast<float*>(ws + zacc_offset(m));
  a.debug_stall = g_debug_stall.load(std::memory_order_relaxed);
  const int path = g_path.load(std::memory_order_relaxed);
  const bool tensor = path == EXL3_PATH_TENSOR || (path == EXL3_PATH_AUTO && M > 2);
  if (tensor) {
    // x-tilde as operand-B images (and, for 1MAD, its block sums), then the
    // persistent tensor-core kernel into zacc, then the output transform; the
    // last two are programmatic dependents of the kernel before them.
    __half* bimg = reinterpret_cast<__half*>(ws + bimg_offset(m, M));
    float* bsum = codebook == EXL3_CB_1MAD ? reinterpret_cast<float*>(ws + bsum_offset(m, n, M)) : nullptr;
    a.y = reinterpret_cast<__half*>(y);
    if ((st = launch_bimg(reinterpret_cast<const __half*>(x), a.s_in, bimg, bsum, M, tc_nb(M), n, cs)) !=
        EXL3_OK)
      return st;
    if ((st = launch_tc(a, bimg, bsum, M, sms, cs)) != EXL3_OK) return st;
    return launch_epi(a.zacc, a.scales, a.s_out, a.y, M, m, cs);
  }
  // x pairs of each batch chunk go where the tensor path keeps its operand
  // images (at least 32 n bytes, enough for 8 rows of n 32-bit pairs).
  uint32_t* xd = reinterpret_cast<uint32_t*>(ws + bimg_offset(m, M));
  for (int done = 0; done < M;) {
    const int rem = M - done;
    const int mb = rem >= 8 ? 8 : rem >= 4 ? 4 : rem >= 2 ? 2 : 1;
    a.x = reinterpret_cast<const __half*>(x) + static_cast<size_t>(done) * n;
    a.y = reinterpret_cast<__half*>(y) + static_cast<size_t>(done) * m;
    const LayerPlan plan = plan_layer(m, n, mb, sms);
    a.ctas = plan.ctas;
    a.sub = plan.sub;
    if (plan.sub > 0) {
      if ((st = launch_xdup(a.x, a.s_in, xd, mb, n, codebook, cs)) != EXL3_OK) return st;
      a.xdup = xd;
    }
    if ((st = launch_layer(a, mb, cs)) != EXL3_OK) return st;
    if ((st = launch_epi(a.zacc, a.scales, a.s_out, a.y, mb, m, cs)) != EXL3_OK) return st;
    done += mb;
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
