// QTIP's whole-vector rotation ("Trellis Quantization" Part eleven: QTIP
// rotates whole rows and columns, EXL3 rotates 128-blocks).
//
// With Sylvester ordering H_{128 B} = H_B (x) H_128, so the whole-vector
// transform of a power-of-two length d = 128 B is the blockwise 128-point
// transform followed by a B-point transform across the blocks (the two
// commute).  The layer entry point therefore wraps the blockwise layer:
//   x' = binary16(H_B-across(s_in (.) x) / sqrt(B)),
//   u  = blockwise layer on x' with unit input signs (its input transform then
//        completes H_n) and the real s_out (applied before the output
//        transform, as the definition wants),
//   y  = binary16(H_B-across(u) / sqrt(B)) over the m outputs.
// Each wrapper step adds one binary16 rounding of an intermediate vector.
//
// rht_whole_kernel (the standalone transform): one CTA per row, the row in
// shared memory as fp32; the blockwise stage (one warp per 128-block, shuffle
// butterflies), then the butterflies across blocks at spans 128, ..., d / 2.
// rht_cross_kernel (the layer's two wrapper steps): the butterflies across
// blocks only, eight CTAs per row.
#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {

namespace {

constexpr int kWholeThreads = 1024;
constexpr int kWholeMax = 32768;  // fp32 row in 128 KB of shared memory

__global__ void __launch_bounds__(kWholeThreads)
    rht_whole_kernel(const __half* __restrict__ in, const __half* __restrict__ signs,
                     __half* __restrict__ out, int d, float scale) {
  extern __shared__ float u[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const size_t row = blockIdx.x;
  const __half* src = in + row * d;
  // one warp per 128-block: signs, 128-point butterflies, into shared memory
  for (int kb = warp; kb < d / kRowBlock; kb += kWholeThreads / 32) {
    const int col = kb * kRowBlock + 4 * lane;
    const uint2 xr = *reinterpret_cast<const uint2*>(src + col);
    const uint2 sr = *reinterpret_cast<const uint2*>(signs + col);
    const __half2 x01 = *reinterpret_cast<const __half2*>(&xr.x);
    const __half2 x23 = *reinterpret_cast<const __half2*>(&xr.y);
    const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
    const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
    float v[4] = {__low2float(x01) * __low2float(s01), __high2float(x01) * __high2float(s01),
                  __low2float(x23) * __low2float(s23), __high2float(x23) * __high2float(s23)};
    fwht128_warp(v, lane);
    *reinterpret_cast<float4*>(&u[col]) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __syncthreads();
  // butterflies across 128-blocks: pair (i, i + h) for every i with bit h clear
  for (int h = kRowBlock; h < d; h <<= 1) {
    for (int p = tid; p < d / 2; p += kWholeThreads) {
      const int i = (p / h) * 2 * h + (p % h);
      const float a = u[i];
      const float b = u[i + h];
      u[i] = a + b;
      u[i + h] = a - b;
    }
    __syncthreads();
  }
  for (int i = 4 * tid; i < d; i += 4 * kWholeThreads) {
    const float4 v = *reinterpret_cast<const float4*>(&u[i]);
    const __half2 o01 = __floats2half2_rn(v.x * scale, v.y * scale);
    const __half2 o23 = __floats2half2_rn(v.z * scale, v.w * scale);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&o01);
    o.y = *reinterpret_cast<const uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(out + row * d + i) = o;
  }
}

// The transform across the 128-blocks alone, spread over CTAs: CTA (row, c)
// takes within-block columns 16c .. 16c + 15 of every block of the row (the
// butterflies across blocks never mix columns), so a row of any length uses
// eight CTAs.  out = binary16(H_B-across(signs (.) in) * scale), B = d / 128,
// for up to EXL3_MAX_GROUP vectors of their own lengths (CTA row index =
// vector * rows + row).
constexpr int kCrossCols = 16;
constexpr int kCrossThreads = 256;

struct CrossGroup {
  const __half* in[EXL3_MAX_GROUP];
  const __half* signs[EXL3_MAX_GROUP];  // NULL: no signs
  __half* out[EXL3_MAX_GROUP];
  int d[EXL3_MAX_GROUP];
  float scale[EXL3_MAX_GROUP];
  int count;
  int rows;
  __half* ones;  // when not NULL, the CTAs of the first row write ones_len unit signs here
  int ones_len;
};

__global__ void __launch_bounds__(kCrossThreads) rht_cross_kernel(const CrossGroup g) {
  __shared__ float u[(kWholeMax / kRowBlock) * kCrossCols];
  const int l = static_cast<int>(blockIdx.x) / g.rows;
  const size_t row = static_cast<size_t>(blockIdx.x) - static_cast<size_t>(l) * g.rows;
  const int d = g.d[l];
  const __half* __restrict__ in = g.in[l];
  const __half* __restrict__ signs = g.signs[l];
  __half* __restrict__ out = g.out[l];
  const float scale = g.scale[l];
  const int nb = d / kRowBlock;
  const int c0 = blockIdx.y * kCrossCols;
  const int tid = threadIdx.x;
  // element e of this CTA: block e / 16, column c0 + e % 16
  for (int e2 = tid; e2 < nb * kCrossCols / 2; e2 += kCrossThreads) {
    const int e = 2 * e2;
    const int col = (e / kCrossCols) * kRowBlock + c0 + (e % kCrossCols);
    const __half2 x = *reinterpret_cast<const __half2*>(in + row * d + col);
    float a = __low2float(x), b = __high2float(x);
    if (signs != nullptr) {
      const __half2 sg = *reinterpret_cast<const __half2*>(signs + col);
      a *= __low2float(sg);
      b *= __high2float(sg);
    }
    u[e] = a;
    u[e + 1] = b;
  }
  __syncthreads();
  for (int h = 1; h < nb; h <<= 1) {
    for (int q = tid; q < nb / 2 * kCrossCols; q += kCrossThreads) {
      const int pr = q / kCrossCols;  // pair of blocks (b, b + h), bit h of b clear
      const int j = q % kCrossCols;
      const int b = (pr / h) * 2 * h + (pr % h);
      const float x0 = u[b * kCrossCols + j];
      const float x1 = u[(b + h) * kCrossCols + j];
      u[b * kCrossCols + j] = x0 + x1;
      u[(b + h) * kCrossCols + j] = x0 - x1;
    }
    __syncthreads();
  }
  for (int e2 = tid; e2 < nb * kCrossCols / 2; e2 += kCrossThreads) {
    const int e = 2 * e2;
    const int col = (e / kCrossCols) * kRowBlock + c0 + (e % kCrossCols);
    *reinterpret_cast<__half2*>(out + row * d + col) = __floats2half2_rn(u[e] * scale, u[e + 1] * scale);
  }
  // the CTAs of the first row also write the inner layers' unit signs
  if (g.ones != nullptr && blockIdx.x == 0)
    for (int i = blockIdx.y * kCrossThreads + tid; i < g.ones_len; i += gridDim.y * kCrossThreads)
      g.ones[i] = __float2half_rn(1.0f);
}

// Adds vector l of a cross-block transform group (scale 1/sqrt(d/128)).
void cross_add(CrossGroup& g, const __half* in, const __half* signs, __half* out, int d) {
  g.in[g.count] = in;
  g.signs[g.count] = signs;
  g.out[g.count] = out;
  g.d[g.count] = d;
  g.scale[g.count] = static_cast<float>(1.0 / sqrt(static_cast<double>(d / kRowBlock)));
  ++g.count;
}

exl3_status launch_cross_group(const CrossGroup& g, cudaStream_t stream) {
  if (g.count == 0) return EXL3_OK;
  rht_cross_kernel<<<dim3(static_cast<unsigned>(g.rows * g.count), kRowBlock / kCrossCols), kCrossThreads, 0,
                     stream>>>(g);
  return launch_status();
}

exl3_status launch_rht_cross(const __half* in, const __half* signs, __half* out, int rows, int d, __half* ones,
                             int ones_len, cudaStream_t stream) {
  CrossGroup g{};
  g.rows = rows;
  g.ones = ones;
  g.ones_len = ones_len;
  cross_add(g, in, signs, out, d);
  return launch_cross_group(g, stream);
}

bool whole_length(int d) { return d >= kRowBlock && d <= kWholeMax && (d & (d - 1)) == 0; }

exl3_status launch_rht_whole(const __half* in, const __half* signs, __half* out, int rows, int d,
                             cudaStream_t stream) {
  const size_t smem = sizeof(float) * static_cast<size_t>(d);
  if (cudaFuncSetAttribute(rht_whole_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sizeof(float) * kWholeMax)) != cudaSuccess)
    return EXL3_ERR_CUDA;
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(d)));
  rht_whole_kernel<<<rows, kWholeThreads, smem, stream>>>(in, signs, out, d, scale);
  return launch_status();
}

inline size_t whole_inner_bytes(int m, int n, int M) { return align256(exl3_gemm_workspace_bytes(m, n, M)); }

}  // namespace

}  // namespace exl3

using namespace exl3;

extern "C" exl3_status exl3_rht_whole(const exl3_half* in, const exl3_half* signs, exl3_half* out, int rows,
                                      int d, exl3_stream_t stream) {
  if (rows < 1) return EXL3_ERR_BATCH;
  if (!whole_length(d)) return EXL3_ERR_SHAPE;
  if (!in || !signs || !out) return EXL3_ERR_NULL;
  if (!aligned16(in) || !aligned16(signs) || !aligned16(out)) return EXL3_ERR_ALIGN;
  return launch_rht_whole(reinterpret_cast<const __half*>(in), reinterpret_cast<const __half*>(signs),
                          reinterpret_cast<__half*>(out), rows, d, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t exl3_gemm_whole_workspace_bytes(int m, int n, int M) {
  if (!whole_length(m) || !whole_length(n) || M < 1) return 0;
  const size_t inner = whole_inner_bytes(m, n, M);
  if (inner == 0) return 0;
  const int ones = m > n ? m : n;
  return inner + align256(sizeof(__half) * static_cast<size_t>(ones)) +
         align256(sizeof(__half) * static_cast<size_t>(M) * n) + align256(sizeof(__half) * static_cast<size_t>(M) * m);
}

extern "C" exl3_status exl3_gemm_whole(const uint32_t* codes, int K, int codebook, int m, int n,
                                       const exl3_half* s_in, const exl3_half* s_out, const exl3_half* scales,
                                       int M, const exl3_half* x, exl3_half* y, void* workspace,
                                       size_t workspace_bytes, exl3_stream_t stream) {
  if (M < 1) return EXL3_ERR_BATCH;
  if (!whole_length(m) || !whole_length(n)) return EXL3_ERR_SHAPE;
  exl3_status st = check_k_cb(K, codebook);
  if (st != EXL3_OK) return st;
  if (!codes || !scales || !x || !y) return EXL3_ERR_NULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(y) || (s_in && !aligned16(s_in)) ||
      (s_out && !aligned16(s_out)))
    return EXL3_ERR_ALIGN;
  if (!workspace || workspace_bytes < exl3_gemm_whole_workspace_bytes(m, n, M)) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // [inner layer workspace | unit signs | x' | u]; the inner workspace comes
  // first so the status word sits where exl3_workspace_bytes puts it.
  char* ws = static_cast<char*>(workspace);
  const size_t inner = whole_inner_bytes(m, n, M);
  __half* ones = reinterpret_cast<__half*>(ws + inner);
  const int ones_len = m > n ? m : n;
  __half* xp = reinterpret_cast<__half*>(ws + inner + align256(sizeof(__half) * static_cast<size_t>(ones_len)));
  __half* up = xp + align256(sizeof(__half) * static_cast<size_t>(M) * n) / sizeof(__half);
  const exl3_half* x_in = x;
  const exl3_half* signs_in = nullptr;
  if (s_in != nullptr) {
    if ((st = launch_rht_cross(reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(s_in), xp, M, n,
                               ones, ones_len, cs)) != EXL3_OK)
      return st;
    x_in = reinterpret_cast<const exl3_half*>(xp);
    signs_in = reinterpret_cast<const exl3_half*>(ones);
  }
  exl3_half* y_inner = s_out != nullptr ? reinterpret_cast<exl3_half*>(up) : y;
  if ((st = exl3_gemm(codes, K, codebook, m, n, signs_in, s_out, scales, M, x_in, y_inner, workspace, inner,
                      stream)) != EXL3_OK)
    return st;
  if (s_out != nullptr) return launch_rht_cross(up, nullptr, reinterpret_cast<__half*>(y), M, m, nullptr, 0, cs);
  return EXL3_OK;
}

extern "C" size_t exl3_gemm_whole_grouped_workspace_bytes(const exl3_layer* layers, int count, int M) {
  if (layers == nullptr || count < 1 || count > EXL3_MAX_GROUP || M < 1 || M > EXL3_MAX_BATCH) return 0;
  int ones = 0;
  size_t vecs = 0;
  for (int i = 0; i < count; ++i) {
    const int m = layers[i].m, n = layers[i].n;
    if (!whole_length(m) || !whole_length(n)) return 0;
    ones = m > ones ? m : ones;
    ones = n > ones ? n : ones;
    vecs += align256(sizeof(__half) * static_cast<size_t>(M) * n) + align256(sizeof(__half) * static_cast<size_t>(M) * m);
  }
  const size_t inner = exl3_group_workspace_bytes(layers, count, M);
  if (inner == 0) return 0;
  return align256(inner) + align256(sizeof(__half) * static_cast<size_t>(ones)) + vecs;
}

extern "C" exl3_status exl3_gemm_whole_grouped(const exl3_layer* layers, int count, int K, int codebook, int M,
                                               void* workspace, size_t workspace_bytes, exl3_stream_t stream) {
  if (layers == nullptr) return EXL3_ERR_NULL;
  if (count < 1 || count > EXL3_MAX_GROUP) return EXL3_ERR_BATCH;  // as exl3_gemm_grouped
  if (M < 1 || M > EXL3_MAX_BATCH) return EXL3_ERR_BATCH;
  for (int i = 0; i < count; ++i)
    if (!whole_length(layers[i].m) || !whole_length(layers[i].n)) return EXL3_ERR_SHAPE;
  exl3_status st = check_k_cb(K, codebook);
  if (st != EXL3_OK) return st;
  for (int i = 0; i < count; ++i) {
    const exl3_layer& L = layers[i];
    if (!L.codes || !L.scales || !L.x || !L.y) return EXL3_ERR_NULL;
    if (!aligned16(L.codes) || !aligned16(L.scales) || !aligned16(L.x) || !aligned16(L.y) ||
        (L.s_in && !aligned16(L.s_in)) || (L.s_out && !aligned16(L.s_out)))
      return EXL3_ERR_ALIGN;
  }
  if (!workspace || workspace_bytes < exl3_gemm_whole_grouped_workspace_bytes(layers, count, M))
    return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // [inner group workspace | unit signs | x' of every layer | u of every layer]
  char* ws = static_cast<char*>(workspace);
  const size_t inner = align256(exl3_group_workspace_bytes(layers, count, M));
  int ones_len = 0;
  for (int i = 0; i < count; ++i) {
    ones_len = layers[i].m > ones_len ? layers[i].m : ones_len;
    ones_len = layers[i].n > ones_len ? layers[i].n : ones_len;
  }
  __half* ones = reinterpret_cast<__half*>(ws + inner);
  char* cur = ws + inner + align256(sizeof(__half) * static_cast<size_t>(ones_len));
  exl3_layer in_layers[EXL3_MAX_GROUP];
  CrossGroup gin{}, gout{};
  gin.rows = gout.rows = M;
  gin.ones = ones;
  gin.ones_len = ones_len;
  for (int i = 0; i < count; ++i) {
    const exl3_layer& L = layers[i];
    __half* xp = reinterpret_cast<__half*>(cur);
    cur += align256(sizeof(__half) * static_cast<size_t>(M) * L.n);
    __half* up = reinterpret_cast<__half*>(cur);
    cur += align256(sizeof(__half) * static_cast<size_t>(M) * L.m);
    in_layers[i] = L;
    if (L.s_in != nullptr) {
      cross_add(gin, reinterpret_cast<const __half*>(L.x), reinterpret_cast<const __half*>(L.s_in), xp, L.n);
      in_layers[i].x = reinterpret_cast<const exl3_half*>(xp);
      in_layers[i].s_in = reinterpret_cast<const exl3_half*>(ones);
    }
    if (L.s_out != nullptr) {
      cross_add(gout, up, nullptr, reinterpret_cast<__half*>(L.y), L.m);
      in_layers[i].y = reinterpret_cast<exl3_half*>(up);
    }
  }
  if ((st = launch_cross_group(gin, cs)) != EXL3_OK) return st;
  if ((st = exl3_gemm_grouped(in_layers, count, K, codebook, M, workspace, inner, stream)) != EXL3_OK) return st;
  return launch_cross_group(gout, cs);
}
