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

// One layer's activations for the preparation kernel: binary16 x (rotated
// here with s_in, or taken as already rotated), or int8 q with its scales;
// optional outputs q_out / qscale_out (the quantizer) and the layer kernel's
// operands q4 / tcorr / cs, with the code's centre and scale C.
struct PrepEntry {
  const __half* x;
  const __half* s_in;
  const int8_t* q_in;
  const float* qscale_in;
  int8_t* q_out;
  float* qscale_out;
  int32_t* q4;
  int32_t* tcorr;
  float* cs;
  int n;
  int centre;
  float C;
  long long job_begin;
};
struct PrepGroup {
  PrepEntry e[kMaxGroup];
  int count;
  int rows;
  int rotate;
  long long jobs;
};

__global__ void __launch_bounds__(kPrepThreads) i8_prep_kernel(const PrepGroup g) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long job = static_cast<long long>(blockIdx.x) * (kPrepThreads / 32) + (threadIdx.x >> 5);
  if (job >= g.jobs) return;
  int li = 0;
  {
    int hi = g.count - 1;  // the last layer whose first job is <= job
    while (li < hi) {
      const int mid = (li + hi + 1) >> 1;
      if (job >= g.e[mid].job_begin) li = mid; else hi = mid - 1;
    }
  }
  const PrepEntry& e = g.e[li];
  const int n = e.n;
  const int nkb = n / kRowBlock;
  const long long local = job - e.job_begin;
  const int row = static_cast<int>(local / nkb);
  const int kb = static_cast<int>(local - static_cast<long long>(row) * nkb);
  const int col = kb * kRowBlock + 4 * lane;
  const size_t at = static_cast<size_t>(row) * n + col;
  int q[4];
  float scale;
  if (e.q_in != nullptr) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(e.q_in + at);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = static_cast<int>(static_cast<int8_t>(w >> (8 * i)));
    scale = e.qscale_in[static_cast<size_t>(row) * nkb + kb];
  } else {
    const uint2 xr = *reinterpret_cast<const uint2*>(e.x + at);
    const __half2 x01 = *reinterpret_cast<const __half2*>(&xr.x);
    const __half2 x23 = *reinterpret_cast<const __half2*>(&xr.y);
    float v[4] = {__low2float(x01), __high2float(x01), __low2float(x23), __high2float(x23)};
    if (g.rotate && e.s_in != nullptr) {
      const uint2 sr = *reinterpret_cast<const uint2*>(e.s_in + col);
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
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
    scale = __fdiv_rn(amax, 127.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = amax > 0.0f ? __float2int_rn(__fdiv_rn(v[i], scale)) : 0;
    if (e.q_out != nullptr) {
      const uint32_t w = (static_cast<uint32_t>(q[0]) & 0xFFu) | ((static_cast<uint32_t>(q[1]) & 0xFFu) << 8) |
                         ((static_cast<uint32_t>(q[2]) & 0xFFu) << 16) | ((static_cast<uint32_t>(q[3]) & 0xFFu) << 24);
      *reinterpret_cast<uint32_t*>(e.q_out + at) = w;
    }
    if (e.qscale_out != nullptr && lane == 0) e.qscale_out[static_cast<size_t>(row) * nkb + kb] = scale;
  }
  if (e.q4 != nullptr) {
    int4 r;
    r.x = static_cast<int>((static_cast<uint32_t>(q[0]) & 0xFFu) * 0x01010101u);
    r.y = static_cast<int>((static_cast<uint32_t>(q[1]) & 0xFFu) * 0x01010101u);
    r.z = static_cast<int>((static_cast<uint32_t>(q[2]) & 0xFFu) * 0x01010101u);
    r.w = static_cast<int>((static_cast<uint32_t>(q[3]) & 0xFFu) * 0x01010101u);
    *reinterpret_cast<int4*>(e.q4 + at) = r;
    // lanes 4t .. 4t + 3 hold the 16 columns of tile t of the block
    int s = q[0] + q[1] + q[2] + q[3];
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
    if ((lane & 3) == 0) e.tcorr[static_cast<size_t>(row) * (n / 16) + col / 16] = e.centre * s;
    if (lane == 0) e.cs[static_cast<size_t>(row) * nkb + kb] = __fmul_rn(e.C, scale);
  }
}

void set_code(PrepEntry& e, int codebook) {
  e.centre = codebook == EXL3_CB_MUL1 ? kMul1Centre : kOneMadCentre;
  e.C = codebook == EXL3_CB_MUL1 ? kMul1Scale : kOneMadScale;
}

// Entries carry their code's centre and scale (set_code).
exl3_status launch_prep(PrepGroup g, cudaStream_t stream) {
  long long jobs = 0;
  for (int i = 0; i < g.count; ++i) {
    g.e[i].job_begin = jobs;
    jobs += static_cast<long long>(g.rows) * (g.e[i].n / kRowBlock);
  }
  g.jobs = jobs;
  const long long per_cta = kPrepThreads / 32;
  const unsigned grid = static_cast<unsigned>((jobs + per_cta - 1) / per_cta);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, i8_prep_kernel, g) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

exl3_status launch_i8_kset(const I8Args& a, int K, cudaStream_t stream) {
  switch (K) {
    case 1: return launch_i8_kset_k1(a, stream);
    case 2: return launch_i8_kset_k2(a, stream);
    case 3: return launch_i8_kset_k3(a, stream);
    case 4: return launch_i8_kset_k4(a, stream);
    case 5: return launch_i8_kset_k5(a, stream);
    case 6: return launch_i8_kset_k6(a, stream);
    case 7: return launch_i8_kset_k7(a, stream);
    default: return launch_i8_kset_k8(a, stream);
  }
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

// Per-layer operands of the int8 path in a workspace: fp32 row sums [M][m],
// q4 [M][n] int32, tile corrections [M][n/16] int32, block factors [M][n/128]
// fp32, each 256-byte aligned, from byte `at`.
struct I8Region {
  float* zacc;
  int32_t* q4;
  int32_t* tcorr;
  float* cs;
};
size_t i8_layer_bytes(int m, int n, int M) {
  return align256(sizeof(float) * static_cast<size_t>(M) * m) + align256(sizeof(int32_t) * static_cast<size_t>(M) * n) +
         align256(sizeof(int32_t) * static_cast<size_t>(M) * (n / 16)) +
         align256(sizeof(float) * static_cast<size_t>(M) * (n / kRowBlock));
}
I8Region i8_region(char* ws, size_t at, int m, int n, int M) {
  I8Region r;
  r.zacc = reinterpret_cast<float*>(ws + at);
  at += align256(sizeof(float) * static_cast<size_t>(M) * m);
  r.q4 = reinterpret_cast<int32_t*>(ws + at);
  at += align256(sizeof(int32_t) * static_cast<size_t>(M) * n);
  r.tcorr = reinterpret_cast<int32_t*>(ws + at);
  at += align256(sizeof(int32_t) * static_cast<size_t>(M) * (n / 16));
  r.cs = reinterpret_cast<float*>(ws + at);
  return r;
}
// Single layer: counters and status word, then the layer's region.
size_t i8_total(int m, int n, int M) { return zacc_offset(m) + i8_layer_bytes(m, n, M); }

exl3_status check_i8(const uint32_t* codes, int K, int codebook, int m, int n, const exl3_half* s_out,
                     const exl3_half* scales, int M, const void* xin, exl3_half* y) {
  if (M < 1 || M > EXL3_MAX_BATCH) return EXL3_ERR_BATCH;
  exl3_status st = check_shape(m, n);
  if (st != EXL3_OK) return st;
  if ((st = check_k_cb(K, codebook)) != EXL3_OK) return st;
  if (codebook != EXL3_CB_1MAD && codebook != EXL3_CB_MUL1) return EXL3_ERR_CODEBOOK;
  if (!codes || !scales || !xin || !y) return EXL3_ERR_NULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(xin) || !aligned16(y) || (s_out && !aligned16(s_out)))
    return EXL3_ERR_ALIGN;
  return EXL3_OK;
}

// Per batch chunk of 8/4/2/1 rows, one layer kernel per (K, code) class over
// that class's layers (classes in order of first appearance; ks / cbs give
// each layer's K and code), then one output kernel over all layers and rows.
exl3_status run_i8(const exl3_layer* layers, const I8Region* reg, int count, const int* ks, const int* cbs, int M,
                   cudaStream_t cs) {
  const int sms = device_sm_count();
  int cls[kMaxGroup], nclass = 0;  // the first layer of each class
  int of[kMaxGroup];               // each layer's class
  long long tiles[kMaxGroup] = {};
  for (int i = 0; i < count; ++i) {
    int c = 0;
    while (c < nclass && (ks[cls[c]] != ks[i] || cbs[cls[c]] != cbs[i])) ++c;
    if (c == nclass) cls[nclass++] = i;
    of[i] = c;
    tiles[c] += static_cast<long long>(layers[i].m / 16) * (layers[i].n / 16);
  }
  exl3_status st;
  for (int done = 0; done < M;) {
    const int mb = M - done >= 8 ? 8 : M - done >= 4 ? 4 : M - done >= 2 ? 2 : 1;
    // layer i's entry of a launch of `sub`-tile sub-units; units counts on
    auto add_layer = [&](I8Args& a, int i, int sub, long long& units) {
      const int m = layers[i].m, n = layers[i].n;
      I8Layer& l = a.l[a.count++];
      l.codes = layers[i].codes;
      l.q4 = reg[i].q4 + static_cast<size_t>(done) * n;
      l.tcorr = reg[i].tcorr + static_cast<size_t>(done) * (n / 16);
      l.cs = reg[i].cs + static_cast<size_t>(done) * (n / kRowBlock);
      l.zacc = reg[i].zacc + static_cast<size_t>(done) * m;
      l.m = m;
      l.n = n;
      l.u_begin = static_cast<int>(units);
      l.per_row = (n / 16 + sub - 1) / sub;
      l.row_magic = div_magic(l.per_row, static_cast<long long>(m / 16) * l.per_row);
      units += static_cast<long long>(m / 16) * l.per_row;
    };
    bool launched[kMaxGroup] = {};
    for (int c = 0; c < nclass; ++c) {
      if (launched[c]) continue;
      const int K = ks[cls[c]];
      if (mb == 1) {
        // both codes of this K: at 32-tile sub-units, one launch
        long long ktiles = 0;
        int nk = 0;
        for (int c2 = c; c2 < nclass; ++c2)
          if (ks[cls[c2]] == K) {
            ktiles += tiles[c2];
            ++nk;
          }
        if (nk > 1 && choose_sub(ktiles, 1, sms) == 32) {
          I8Args a{};
          a.sub = 32;
          long long units = 0;
          const int order[2] = {EXL3_CB_1MAD, EXL3_CB_MUL1};
          for (int k = 0; k < 2; ++k) {
            for (int i = 0; i < count; ++i)
              if (ks[i] == K && cbs[i] == order[k]) add_layer(a, i, 32, units);
            a.class_end[k] = units;
          }
          a.units = units;
          a.ctas = static_cast<int>(units < sms ? units : sms);
          if ((st = launch_i8_kset(a, K, cs)) != EXL3_OK) return st;
          for (int c2 = c; c2 < nclass; ++c2)
            if (ks[cls[c2]] == K) launched[c2] = true;
          continue;
        }
      }
      I8Args a{};
      a.sub = choose_sub(tiles[c], mb, sms);
      long long units = 0;
      for (int i = 0; i < count; ++i)
        if (of[i] == c) add_layer(a, i, a.sub, units);
      a.units = units;
      a.ctas = static_cast<int>(units < sms ? units : sms);
      if ((st = launch_i8(a, K, cbs[cls[c]], mb, cs)) != EXL3_OK) return st;
    }
    done += mb;
  }
  EpiGroup eg{};
  eg.count = count;
  eg.rows = M;
  for (int i = 0; i < count; ++i) {
    eg.e[i].zacc = reg[i].zacc;
    eg.e[i].scales = reinterpret_cast<const __half*>(layers[i].scales);
    eg.e[i].s_out = reinterpret_cast<const __half*>(layers[i].s_out);
    eg.e[i].y = reinterpret_cast<__half*>(layers[i].y);
    eg.e[i].m = layers[i].m;
  }
  return launch_epi_group(eg, cs);
}

exl3_layer layer_of(const uint32_t* codes, int m, int n, const exl3_half* s_in, const exl3_half* s_out,
                    const exl3_half* scales, const exl3_half* x, exl3_half* y) {
  exl3_layer L{};
  L.codes = codes;
  L.m = m;
  L.n = n;
  L.s_in = s_in;
  L.s_out = s_out;
  L.scales = scales;
  L.x = x;
  L.y = y;
  return L;
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
  PrepGroup g{};
  g.count = 1;
  g.rows = M;
  g.rotate = 0;
  g.e[0].x = reinterpret_cast<const __half*>(x_rot);
  g.e[0].q_out = q;
  g.e[0].qscale_out = qscale;
  g.e[0].n = n;
  return launch_prep(g, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t exl3_gemm_i8_workspace_bytes(int m, int n, int M) {
  if (check_shape(m, n) != EXL3_OK || M < 1 || M > EXL3_MAX_BATCH) return 0;
  return i8_total(m, n, M);
}

extern "C" exl3_status exl3_gemm_i8(const uint32_t* codes, int K, int codebook, int m, int n,
                                    const exl3_half* s_out, const exl3_half* scales, int M, const int8_t* q,
                                    const float* qscale, exl3_half* y, void* workspace, size_t workspace_bytes,
                                    exl3_stream_t stream) {
  exl3_status st = check_i8(codes, K, codebook, m, n, s_out, scales, M, q, y);
  if (st != EXL3_OK) return st;
  if (!qscale) return EXL3_ERR_NULL;
  if (!workspace || workspace_bytes < i8_total(m, n, M)) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const I8Region reg = i8_region(ws, zacc_offset(m), m, n, M);
  PrepGroup g{};
  g.count = 1;
  g.rows = M;
  g.e[0].q_in = q;
  g.e[0].qscale_in = qscale;
  g.e[0].q4 = reg.q4;
  g.e[0].tcorr = reg.tcorr;
  g.e[0].cs = reg.cs;
  g.e[0].n = n;
  set_code(g.e[0], codebook);
  if ((st = launch_prep(g, cs)) != EXL3_OK) return st;
  const exl3_layer L = layer_of(codes, m, n, nullptr, s_out, scales, nullptr, y);
  return run_i8(&L, &reg, 1, &K, &codebook, M, cs);
}

// x of every layer rotated and quantized in one preparation kernel, then the
// layer kernels and the output kernel over the whole group.
exl3_status run_int8act(const exl3_layer* layers, const I8Region* reg, int count, const int* ks, const int* cbs,
                        int M, cudaStream_t cs) {
  PrepGroup g{};
  g.count = count;
  g.rows = M;
  g.rotate = 1;
  for (int i = 0; i < count; ++i) {
    g.e[i].x = reinterpret_cast<const __half*>(layers[i].x);
    g.e[i].s_in = reinterpret_cast<const __half*>(layers[i].s_in);
    g.e[i].q4 = reg[i].q4;
    g.e[i].tcorr = reg[i].tcorr;
    g.e[i].cs = reg[i].cs;
    g.e[i].n = layers[i].n;
    set_code(g.e[i], cbs[i]);
  }
  exl3_status st = launch_prep(g, cs);
  if (st != EXL3_OK) return st;
  return run_i8(layers, reg, count, ks, cbs, M, cs);
}

extern "C" exl3_status exl3_gemm_int8act(const uint32_t* codes, int K, int codebook, int m, int n,
                                         const exl3_half* s_in, const exl3_half* s_out, const exl3_half* scales,
                                         int M, const exl3_half* x, exl3_half* y, void* workspace,
                                         size_t workspace_bytes, exl3_stream_t stream) {
  exl3_status st = check_i8(codes, K, codebook, m, n, s_out, scales, M, x, y);
  if (st != EXL3_OK) return st;
  if (s_in && !aligned16(s_in)) return EXL3_ERR_ALIGN;
  if (!workspace || workspace_bytes < i8_total(m, n, M)) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;
  const I8Region reg = i8_region(static_cast<char*>(workspace), zacc_offset(m), m, n, M);
  const exl3_layer L = layer_of(codes, m, n, s_in, s_out, scales, x, y);
  return run_int8act(&L, &reg, 1, &K, &codebook, M, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t exl3_group_i8_workspace_bytes(const exl3_layer* layers, int count, int M) {
  if (layers == nullptr || count < 1 || count > EXL3_MAX_GROUP || M < 1 || M > EXL3_MAX_BATCH) return 0;
  size_t b = 256;  // the status word
  for (int i = 0; i < count; ++i) {
    if (check_shape(layers[i].m, layers[i].n) != EXL3_OK) return 0;
    b += i8_layer_bytes(layers[i].m, layers[i].n, M);
  }
  return b;
}

extern "C" exl3_status exl3_gemm_int8act_grouped(const exl3_layer* layers, int count, int K, int codebook, int M,
                                                 void* workspace, size_t workspace_bytes, exl3_stream_t stream) {
  if (layers == nullptr) return EXL3_ERR_NULL;
  if (count < 1 || count > EXL3_MAX_GROUP) return EXL3_ERR_BATCH;
  exl3_status st;
  for (int i = 0; i < count; ++i) {
    const exl3_layer& L = layers[i];
    if ((st = check_i8(L.codes, K, codebook, L.m, L.n, L.s_out, L.scales, M, L.x, L.y)) != EXL3_OK) return st;
    if (L.s_in && !aligned16(L.s_in)) return EXL3_ERR_ALIGN;
  }
  const size_t need = exl3_group_i8_workspace_bytes(layers, count, M);
  if (!workspace || workspace_bytes < need) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;
  char* ws = static_cast<char*>(workspace);
  I8Region reg[kMaxGroup];
  int ks[kMaxGroup], cbs[kMaxGroup];
  size_t at = 256;
  for (int i = 0; i < count; ++i) {
    reg[i] = i8_region(ws, at, layers[i].m, layers[i].n, M);
    at += i8_layer_bytes(layers[i].m, layers[i].n, M);
    ks[i] = K;
    cbs[i] = codebook;
  }
  return run_int8act(layers, reg, count, ks, cbs, M, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t exl3_multi_i8_workspace_bytes(const exl3_layer_kc* layers, int count, int M) {
  if (layers == nullptr || count < 1 || count > EXL3_MAX_GROUP) return 0;
  exl3_layer plain[kMaxGroup];
  for (int i = 0; i < count; ++i) plain[i] = layers[i].layer;
  return exl3_group_i8_workspace_bytes(plain, count, M);
}

extern "C" exl3_status exl3_gemm_int8act_multi(const exl3_layer_kc* layers, int count, int M, void* workspace,
                                               size_t workspace_bytes, exl3_stream_t stream) {
  if (layers == nullptr) return EXL3_ERR_NULL;
  if (count < 1 || count > EXL3_MAX_GROUP) return EXL3_ERR_BATCH;
  exl3_layer plain[kMaxGroup];
  int ks[kMaxGroup], cbs[kMaxGroup];
  exl3_status st;
  for (int i = 0; i < count; ++i) {
    const exl3_layer& L = layers[i].layer;
    if ((st = check_i8(L.codes, layers[i].K, layers[i].codebook, L.m, L.n, L.s_out, L.scales, M, L.x, L.y)) !=
        EXL3_OK)
      return st;
    if (L.s_in && !aligned16(L.s_in)) return EXL3_ERR_ALIGN;
    plain[i] = L;
    ks[i] = layers[i].K;
    cbs[i] = layers[i].codebook;
  }
  const size_t need = exl3_group_i8_workspace_bytes(plain, count, M);
  if (!workspace || workspace_bytes < need) return EXL3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXL3_ERR_ALIGN;
  char* ws = static_cast<char*>(workspace);
  I8Region reg[kMaxGroup];
  size_t at = 256;
  for (int i = 0; i < count; ++i) {
    reg[i] = i8_region(ws, at, plain[i].m, plain[i].n, M);
    at += i8_layer_bytes(plain[i].m, plain[i].n, M);
  }
  return run_int8act(plain, reg, count, ks, cbs, M, reinterpret_cast<cudaStream_t>(stream));
}
