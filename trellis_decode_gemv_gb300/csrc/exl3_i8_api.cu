// The int8-activation path's host entry points and its small kernels
// ("Trellis Quantization" Part eleven: quantize the activations to eight-bit
// integers and fuse the byte-sum decode with the multiply in one dp4a).
//
// Activation quantization (the pages do not give it; reading): symmetric, per
// 128-column block of each row of the rotated activations x-tilde in
// binary16, in binary32: scale = max|x| / 127, q = nearest integer to
// x / scale (ties to even), both divisions correctly rounded; a block of
// zeros has scale 0 and q 0.
//
// i8_prep_kernel, one warp per (row, 128-block), four columns per lane:
//   optional input transform x-tilde = binary16(Hb(s_in (.) x) / sqrt(128)),
//   or the int8 activations and scales given by the caller;
//   the quantization above;
//   for the layer kernel: each q replicated into the four bytes of a word,
//   centre x the sum of q over each 16-column tile, C x scale per block.
#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {

namespace {

constexpr int kPrepThreads = 128;

__global__ void __launch_bounds__(kPrepThreads)
    i8_prep_kernel(const __half* __restrict__ x, const __half* __restrict__ s_in, int rotate,
                   const int8_t* __restrict__ q_in, const float* __restrict__ qscale_in, int8_t* __restrict__ q_out,
                   float* __restrict__ qscale_out, int32_t* __restrict__ q4, int32_t* __restrict__ tcorr,
                   float* __restrict__ cs, int rows, int n, int centre, float C) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int nkb = n / kRowBlock;
  const long long job = static_cast<long long>(blockIdx.x) * (kPrepThreads / 32) + (threadIdx.x >> 5);
  if (job >= static_cast<long long>(rows) * nkb) return;
  const int row = static_cast<int>(job / nkb);
  const int kb = static_cast<int>(job - static_cast<long long>(row) * nkb);
  const int col = kb * kRowBlock + 4 * lane;
  const size_t at = static_cast<size_t>(row) * n + col;
  int q[4];
  float scale;
  if (q_in != nullptr) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(q_in + at);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = static_cast<int>(static_cast<int8_t>(w >> (8 * i)));
    scale = qscale_in[static_cast<size_t>(row) * nkb + kb];
  } else {
    const uint2 xr = *reinterpret_cast<const uint2*>(x + at);
    const __half2 x01 = *reinterpret_cast<const __half2*>(&xr.x);
    const __half2 x23 = *reinterpret_cast<const __half2*>(&xr.y);
    float v[4] = {__low2float(x01), __high2float(x01), __low2float(x23), __high2float(x23)};
    if (rotate) {
      if (s_in != nullptr) {
        const uint2 sr = *reinterpret_cast<const uint2*>(s_in + col);
        const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
        const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
        v[0] *= __low2float(s01);
        v[1] *= __high2float(s01);
        v[2] *= __low2float(s23);
        v[3] *= __high2float(s23);
        fwht128_warp(v, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __half2float(__float2half_rn(v[i] * kInvSqrt128));
      }
    }
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
    scale = __fdiv_rn(amax, 127.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = amax > 0.0f ? __float2int_rn(__fdiv_rn(v[i], scale)) : 0;
    if (q_out != nullptr) {
      const uint32_t w = (static_cast<uint32_t>(q[0]) & 0xFFu) | ((static_cast<uint32_t>(q[1]) & 0xFFu) << 8) |
                         ((static_cast<uint32_t>(q[2]) & 0xFFu) << 16) | ((static_cast<uint32_t>(q[3]) & 0xFFu) << 24);
      *reinterpret_cast<uint32_t*>(q_out + at) = w;
    }
    if (qscale_out != nullptr && lane == 0) qscale_out[static_cast<size_t>(row) * nkb + kb] = scale;
  }
  if (q4 != nullptr) {
    int4 r;
    r.x = static_cast<int>((static_cast<uint32_t>(q[0]) & 0xFFu) * 0x01010101u);
    r.y = static_cast<int>((static_cast<uint32_t>(q[1]) & 0xFFu) * 0x01010101u);
    r.z = static_cast<int>((static_cast<uint32_t>(q[2]) & 0xFFu) * 0x01010101u);
    r.w = static_cast<int>((static_cast<uint32_t>(q[3]) & 0xFFu) * 0x01010101u);
    *reinterpret_cast<int4*>(q4 + at) = r;
    // lanes 4t .. 4t + 3 hold the 16 columns of tile t of the block
    int s = q[0] + q[1] + q[2] + q[3];
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
    if ((lane & 3) == 0) tcorr[static_cast<size_t>(row) * (n / 16) + col / 16] = centre * s;
    if (lane == 0) cs[static_cast<size_t>(row) * nkb + kb] = __fmul_rn(C, scale);
  }
}

exl3_status launch_prep(const __half* x, const __half* s_in, bool rotate, const int8_t* q_in,
                        const float* qscale_in, int8_t* q_out, float* qscale_out, int32_t* q4, int32_t* tcorr,
                        float* cs, int rows, int n, int codebook, cudaStream_t stream) {
  const long long jobs = static_cast<long long>(rows) * (n / kRowBlock);
  const long long per_cta = kPrepThreads / 32;
  const unsigned grid = static_cast<unsigned>((jobs + per_cta - 1) / per_cta);
  const int centre = codebook == EXL3_CB_MUL1 ? kMul1Centre : kOneMadCentre;
  const float C = codebook == EXL3_CB_MUL1 ? kMul1Scale : kOneMadScale;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, i8_prep_kernel, x, s_in, rotate ? 1 : 0, q_in, qscale_in, q_out, qscale_out, q4,
                         tcorr, cs, rows, n, centre, C) != cudaSuccess)
    return EXL3_ERR_CUDA;
  return launch_status();
}

exl3_status launch_i8(const I8Args& a, int K, int codebook, int mb, cudaStream_t stream) {
  switch (K) {
    case 1: return launch_i8_k1(a, codebook, mb, stream);
    case 2: return launch_i8_k2(a, codebook, mb, stream);
    case 3: return launch_i8_k3(a, codebook, mb, stream);
    case 4: return launch_i8_k4(a, codebook, mb, stream);
    case 5: return launch_i8_k5(a, codebook, mb, stream);
    case 6: return launch_i8_k6(a, codebook, mb, stream);
    case 7: return launch_i8_k7(a, codebook, mb, stream);
    default: return launch_i8_k8(a, codebook, mb, stream);
  }
}

// Workspace: counters and status | fp32 row sums [M][m] | q4 [M][n] int32 |
// tile corrections [M][n/16] int32 | block factors [M][n/128] fp32.
size_t i8_q4_offset(int m, int M) { return zacc_offset(m) + align256(sizeof(float) * static_cast<size_t>(M) * m); }
size_t i8_tcorr_offset(int m, int n, int M) {
  return i8_q4_offset(m, M) + align256(sizeof(int32_t) * static_cast<size_t>(M) * n);
}
size_t i8_cs_offset(int m, int n, int M) {
  return i8_tcorr_offset(m, n, M) + align256(sizeof(int32_t) * static_cast<size_t>(M) * (n / 16));
}
size_t i8_total(int m, int n, int M) {
  return i8_cs_offset(m, n, M) + align256(sizeof(float) * static_cast<size_t>(M) * (n / kRowBlock));
}

exl3_status check_i8(const uint32_t* codes, int K, int codebook, int m, int n, const exl3_half* s_out,
                     const exl3_half* scales, int M, const void* xin, exl3_half* y, void* ws, size_t ws_bytes) {
  if (M < 1 || M > EXL3_MAX_BATCH) return EXL3_ERR_BATCH;
  exl3_status st = check_shape(m, n);
  if (st != EXL3_OK) return st;
  if ((st = check_k_cb(K, codebook)) != EXL3_OK) return st;
  if (codebook != EXL3_CB_1MAD && codebook != EXL3_CB_MUL1) return EXL3_ERR_CODEBOOK;
  if (!codes || !scales || !xin || !y) return EXL3_ERR_NULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(xin) || !aligned16(y) || (s_out && !aligned16(s_out)))
    return EXL3_ERR_ALIGN;
  if (!ws || ws_bytes < i8_total(m, n, M)) return EXL3_ERR_WORKSPACE;
  if (!aligned16(ws)) return EXL3_ERR_ALIGN;
  return EXL3_OK;
}

// The layer kernel per batch chunk of 8/4/2/1 rows, then the output kernel
// over all M rows.
exl3_status run_i8(const uint32_t* codes, int K, int codebook, int m, int n, const __half* s_out,
                   const __half* scales, int M, __half* y, char* ws, cudaStream_t cs) {
  const int sms = device_sm_count();
  float* zacc = reinterpret_cast<float*>(ws + zacc_offset(m));
  const int32_t* q4 = reinterpret_cast<const int32_t*>(ws + i8_q4_offset(m, M));
  const int32_t* tcorr = reinterpret_cast<const int32_t*>(ws + i8_tcorr_offset(m, n, M));
  const float* csb = reinterpret_cast<const float*>(ws + i8_cs_offset(m, n, M));
  const long long tiles = static_cast<long long>(m / 16) * (n / 16);
  exl3_status st;
  for (int done = 0; done < M;) {
    const int mb = M - done >= 8 ? 8 : M - done >= 4 ? 4 : M - done >= 2 ? 2 : 1;
    I8Args a{};
    a.codes = codes;
    a.q4 = q4 + static_cast<size_t>(done) * n;
    a.tcorr = tcorr + static_cast<size_t>(done) * (n / 16);
    a.cs = csb + static_cast<size_t>(done) * (n / kRowBlock);
    a.zacc = zacc + static_cast<size_t>(done) * m;
    a.m = m;
    a.n = n;
    a.sub = choose_sub(tiles, mb, sms);
    a.per_row = (n / 16 + a.sub - 1) / a.sub;
    a.units = static_cast<long long>(m / 16) * a.per_row;
    a.ctas = static_cast<int>(a.units < sms ? a.units : sms);
    if ((st = launch_i8(a, K, codebook, mb, cs)) != EXL3_OK) return st;
    done += mb;
  }
  return launch_epi(zacc, scales, s_out, y, M, m, cs);
}

}  // namespace

}  // namespace exl3

using namespace exl3;

extern "C" exl3_status exl3_quantize_act(const exl3_half* x_rot, int M, int n, int8_t* q, float* qscale,
                                         exl3_stream_t stream) {
  if (M < 1) return EXL3_ERR_BATCH;
  if (n <= 0 || n % kRowBlock) return EXL3_ERR_SHAPE;
  if (!x_rot || !q || !qscale) return EXL3_ERR_NULL;
  if (!aligned16(x_rot) || !aligned16(q)) return EXL3_ERR_ALIGN;
  return launch_prep(reinterpret_cast<const __half*>(x_rot), nullptr, false, nullptr, nullptr, q, qscale, nullptr,
                     nullptr, nullptr, M, n, EXL3_CB_MUL1, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t exl3_gemm_i8_workspace_bytes(int m, int n, int M) {
  if (check_shape(m, n) != EXL3_OK || M < 1 || M > EXL3_MAX_BATCH) return 0;
  return i8_total(m, n, M);
}

extern "C" exl3_status exl3_gemm_i8(const uint32_t* codes, int K, int codebook, int m, int n,
                                    const exl3_half* s_out, const exl3_half* scales, int M, const int8_t* q,
                                    const float* qscale, exl3_half* y, void* workspace, size_t workspace_bytes,
                                    exl3_stream_t stream) {
  exl3_status st = check_i8(codes, K, codebook, m, n, s_out, scales, M, q, y, workspace, workspace_bytes);
  if (st != EXL3_OK) return st;
  if (!qscale) return EXL3_ERR_NULL;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if ((st = launch_prep(nullptr, nullptr, false, q, qscale, nullptr, nullptr,
                        reinterpret_cast<int32_t*>(ws + i8_q4_offset(m, M)),
                        reinterpret_cast<int32_t*>(ws + i8_tcorr_offset(m, n, M)),
                        reinterpret_cast<float*>(ws + i8_cs_offset(m, n, M)), M, n, codebook, cs)) != EXL3_OK)
    return st;
  return run_i8(codes, K, codebook, m, n, reinterpret_cast<const __half*>(s_out),
                reinterpret_cast<const __half*>(scales), M, reinterpret_cast<__half*>(y), ws, cs);
}

extern "C" exl3_status exl3_gemm_int8act(const uint32_t* codes, int K, int codebook, int m, int n,
                                         const exl3_half* s_in, const exl3_half* s_out, const exl3_half* scales,
                                         int M, const exl3_half* x, exl3_half* y, void* workspace,
                                         size_t workspace_bytes, exl3_stream_t stream) {
  exl3_status st = check_i8(codes, K, codebook, m, n, s_out, scales, M, x, y, workspace, workspace_bytes);
  if (st != EXL3_OK) return st;
  if (s_in && !aligned16(s_in)) return EXL3_ERR_ALIGN;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if ((st = launch_prep(reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(s_in), true, nullptr,
                        nullptr, nullptr, nullptr, reinterpret_cast<int32_t*>(ws + i8_q4_offset(m, M)),
                        reinterpret_cast<int32_t*>(ws + i8_tcorr_offset(m, n, M)),
                        reinterpret_cast<float*>(ws + i8_cs_offset(m, n, M)), M, n, codebook, cs)) != EXL3_OK)
    return st;
  return run_i8(codes, K, codebook, m, n, reinterpret_cast<const __half*>(s_out),
                reinterpret_cast<const __half*>(scales), M, reinterpret_cast<__half*>(y), ws, cs);
}
