// Standalone randomized Hadamard transform and tile decode kernels.
//
// rht:    out[r] = Hb(s (.) in[r]) for each row r, Hb = blockwise 128-point
//         Walsh-Hadamard / sqrt(128) ("ExLlamaV3 & EXL3 Deep Dive" Section 2;
//         "Trellis Quantization" Part eleven for the 128-wide blocks).  One
//         warp per 128-block, 4 elements per lane, shuffle butterflies.
// decode: W-hat[16I + r][16J + c] = code(state of step 16r + c of tile (I, J))
//         ("Trellis Quantization" Parts eight and nine).  One thread per row
//         pair of a tile (32 trellis steps), bit-exact binary16 output.
#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {

namespace {

constexpr int kThreads = 256;
// The two small kernels chained to the layer kernels by programmatic dependent
// launch: 128 threads and at most 32 registers, so that a CTA fits beside the
// resident layer kernel and is ready when it finishes.
constexpr int kSmallThreads = 128;

__global__ void __launch_bounds__(kThreads)
    rht_kernel(const __half* __restrict__ in, const __half* __restrict__ signs,
               __half* __restrict__ out, long long blocks, int d) {
  const int lane = threadIdx.x & 31;
  const long long job = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  if (job >= blocks) return;
  const int per_row = d / kRowBlock;
  const long long row = job / per_row;
  const int kb = static_cast<int>(job - row * per_row);
  const int col = kb * kRowBlock + 4 * lane;
  const uint2 xr = *reinterpret_cast<const uint2*>(in + row * d + col);
  const uint2 sr = *reinterpret_cast<const uint2*>(signs + col);
  float v[4];
  {
    const __half2 x01 = *reinterpret_cast<const __half2*>(&xr.x);
    const __half2 x23 = *reinterpret_cast<const __half2*>(&xr.y);
    const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
    const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
    v[0] = __low2float(x01) * __low2float(s01);
    v[1] = __high2float(x01) * __high2float(s01);
    v[2] = __low2float(x23) * __low2float(s23);
    v[3] = __high2float(x23) * __high2float(s23);
  }
  fwht128_warp(v, lane);
  const __half2 o01 = __floats2half2_rn(v[0] * kInvSqrt128, v[1] * kInvSqrt128);
  const __half2 o23 = __floats2half2_rn(v[2] * kInvSqrt128, v[3] * kInvSqrt128);
  uint2 orr;
  orr.x = *reinterpret_cast<const uint32_t*>(&o01);
  orr.y = *reinterpret_cast<const uint32_t*>(&o23);
  *reinterpret_cast<uint2*>(out + row * d + col) = orr;
}

// Operand B images of the tensor-core kernels, for a group of layers.  The M
// batch rows form tiles of nb rows; tile t's image starts at half offset t *
// nb * n.  One warp per (layer, batch row, 128-column block kb): x-tilde =
// Hb(s_in (.) x) of that block (x itself without s_in), rounded to binary16 and
// stored in the canonical K-major no-swizzle layout of an nb x 128 operand:
// element (r, k), r the row within its tile, at half offset ((k / 8) * (nb /
// 8) + r / 8) * 64 + (r % 8) * 8 + k % 8 of the block's image at kb * nb * 128.
// Rows past M are zero.  With bsum, also the fp32 sum of the block's binary16
// values.  Launched as a programmatic dependent (it waits for the preceding
// grid before reading x); the MMA kernels are programmatic dependents of this
// one and wait for it before reading the images.  One launch serves every
// layer of a call (tiles of 128 rows and more use bimg8_kernel below).
__global__ void __launch_bounds__(kSmallThreads, 16) bimg_kernel(const BimgGroup g) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // x may be written by the preceding grid on the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long job = static_cast<long long>(blockIdx.x) * (kSmallThreads / 32) + (threadIdx.x >> 5);
  if (job >= g.jobs) return;
  int li = 0;
  {
    int hi = g.count - 1;  // the last layer whose first job is <= job
    while (li < hi) {
      const int mid = (li + hi + 1) >> 1;
      if (job >= g.e[mid].job_begin) li = mid; else hi = mid - 1;
    }
  }
  const BimgEntry& e = g.e[li];
  const int n = e.n, nb = g.nb, M = g.M;
  const int nkb = n / kRowBlock;
  const long long lj = job - e.job_begin;
  const int gr = static_cast<int>(lj / nkb);  // batch row
  const int kb = static_cast<int>(lj - static_cast<long long>(gr) * nkb);
  const int col = kb * kRowBlock + 4 * lane;
  const uint2 xr = gr < M ? *reinterpret_cast<const uint2*>(e.x + static_cast<size_t>(gr) * n + col)
                          : make_uint2(0u, 0u);
  const int tile = gr / nb;
  const int r = gr - tile * nb;  // row within its tile
  uint2 o = make_uint2(0u, 0u);
  if (gr < M) {  // warp-uniform
    if (e.s_in != nullptr) {
      const uint2 sr = *reinterpret_cast<const uint2*>(e.s_in + col);
      const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
      const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
      const __half2 x01 = *reinterpret_cast<const __half2*>(&xr.x);
      const __half2 x23 = *reinterpret_cast<const __half2*>(&xr.y);
      float v[4] = {__low2float(x01) * __low2float(s01), __high2float(x01) * __high2float(s01),
                    __low2float(x23) * __low2float(s23), __high2float(x23) * __high2float(s23)};
      fwht128_warp(v, lane);
      const __half2 o01 = __floats2half2_rn(v[0] * kInvSqrt128, v[1] * kInvSqrt128);
      const __half2 o23 = __floats2half2_rn(v[2] * kInvSqrt128, v[3] * kInvSqrt128);
      o.x = *reinterpret_cast<const uint32_t*>(&o01);
      o.y = *reinterpret_cast<const uint32_t*>(&o23);
    } else {
      o = xr;
    }
    if (e.bsum != nullptr) {
      const __half2 o01 = *reinterpret_cast<const __half2*>(&o.x);
      const __half2 o23 = *reinterpret_cast<const __half2*>(&o.y);
      float hs = (__low2float(o01) + __high2float(o01)) + (__low2float(o23) + __high2float(o23));
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) hs += __shfl_xor_sync(0xFFFFFFFFu, hs, d);
      if (lane == 0) e.bsum[static_cast<size_t>(gr) * nkb + kb] = hs;
    }
  }
  // This lane's four values are k = 4 * lane .. 4 * lane + 3 of the block.
  const size_t off = static_cast<size_t>(tile) * nb * n + static_cast<size_t>(kb) * nb * kRowBlock +
                     (static_cast<size_t>(lane / 2) * (nb / 8) + r / 8) * 64 + (r % 8) * 8 + (lane % 2) * 4;
  *reinterpret_cast<uint2*>(e.bimg + off) = o;
}

// The same images for tiles of at least 128 rows, eight rows per warp: the
// eight rows of one 8-row group give, per 8-column group, one whole 128-byte
// run of the image, so the warp regroups its rows through shared memory and
// each store instruction writes four whole runs (per-row stores would write
// every 32-byte sector in two halves).
__global__ void __launch_bounds__(kSmallThreads, 8)
    bimg8_kernel(const __half* __restrict__ x, const __half* __restrict__ signs, __half* __restrict__ bimg,
                 float* __restrict__ bsum, int M, int nb, int n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ uint2 runs[kSmallThreads / 32][16 * 8 * 2];  // [8-column group][row][half of the group]
  const int lane = threadIdx.x & 31;
  uint2* run = runs[threadIdx.x >> 5];
  const int nkb = n / kRowBlock;
  const long long job = static_cast<long long>(blockIdx.x) * (kSmallThreads / 32) + (threadIdx.x >> 5);
  const int tiles = (M + nb - 1) / nb;
  if (job >= static_cast<long long>(tiles) * (nb / 8) * nkb) return;
  const int g0 = 8 * static_cast<int>(job / nkb);  // first of eight batch rows, one 8-row group
  const int kb = static_cast<int>(job - static_cast<long long>(g0 / 8) * nkb);
  const int col = kb * kRowBlock + 4 * lane;
  uint2 xr[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    xr[i] = g0 + i < M ? *reinterpret_cast<const uint2*>(x + static_cast<size_t>(g0 + i) * n + col)
                       : make_uint2(0u, 0u);
  float s[4] = {1.f, 1.f, 1.f, 1.f};
  if (signs != nullptr) {
    const uint2 sr = *reinterpret_cast<const uint2*>(signs + col);
    const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
    const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
    s[0] = __low2float(s01);
    s[1] = __high2float(s01);
    s[2] = __low2float(s23);
    s[3] = __high2float(s23);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int g = g0 + i;
    uint2 o = make_uint2(0u, 0u);
    if (g < M) {  // warp-uniform
      if (signs != nullptr) {
        const __half2 x01 = *reinterpret_cast<const __half2*>(&xr[i].x);
        const __half2 x23 = *reinterpret_cast<const __half2*>(&xr[i].y);
        float v[4] = {__low2float(x01) * s[0], __high2float(x01) * s[1], __low2float(x23) * s[2],
                      __high2float(x23) * s[3]};
        fwht128_warp(v, lane);
        const __half2 o01 = __floats2half2_rn(v[0] * kInvSqrt128, v[1] * kInvSqrt128);
        const __half2 o23 = __floats2half2_rn(v[2] * kInvSqrt128, v[3] * kInvSqrt128);
        o.x = *reinterpret_cast<const uint32_t*>(&o01);
        o.y = *reinterpret_cast<const uint32_t*>(&o23);
      } else {
        o = xr[i];
      }
      if (bsum != nullptr) {
        const __half2 o01 = *reinterpret_cast<const __half2*>(&o.x);
        const __half2 o23 = *reinterpret_cast<const __half2*>(&o.y);
        float hs = (__low2float(o01) + __high2float(o01)) + (__low2float(o23) + __high2float(o23));
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) hs += __shfl_xor_sync(0xFFFFFFFFu, hs, d);
        if (lane == 0) bsum[static_cast<size_t>(g) * nkb + kb] = hs;
      }
    }
    // this lane's columns 4 * lane .. + 3 are half (lane % 2) of 8-column group lane / 2
    run[((lane / 2) * 8 + i) * 2 + (lane % 2)] = o;
  }
  __syncwarp();
  // run kg (rows 0..7 of the group, 16 bytes each) lies at half offset
  // (kg * (nb / 8) + r / 8) * 64 of the block image, r the group's first row
  const int tile = g0 / nb;
  const int r = g0 - tile * nb;
  __half* img = bimg + static_cast<size_t>(tile) * nb * n + static_cast<size_t>(kb) * nb * kRowBlock;
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int c = 32 * st + lane;  // 16-byte piece: run c / 8, row c % 8
    const int kg = c / 8;
    const uint4 v = *reinterpret_cast<const uint4*>(&run[2 * c]);
    *reinterpret_cast<uint4*>(img + (static_cast<size_t>(kg) * (nb / 8) + r / 8) * 64 + (c % 8) * 8) = v;
  }
}

// x pairs of the warp-shuffle layer kernel, for a group of layers.  One warp
// per (layer, row, 128-block): x-tilde = Hb(s_in (.) x) / sqrt(128) (x itself
// without s_in), times the code's x factor, rounded once to binary16 and
// duplicated into both halves of a 32-bit word.
__global__ void __launch_bounds__(kSmallThreads, 16) xdup_kernel(const XdupGroup g) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long job = static_cast<long long>(blockIdx.x) * (kSmallThreads / 32) + (threadIdx.x >> 5);
  if (job >= g.jobs) return;
  int li = 0;
  {
    int hi = g.count - 1;  // the last layer whose first job is <= job
    while (li < hi) {
      const int mid = (li + hi + 1) >> 1;
      if (job >= g.e[mid].job_begin) li = mid; else hi = mid - 1;
    }
  }
  const XdupEntry& e = g.e[li];
  const int n = e.n;
  const int per_row = n / kRowBlock;
  const long long local = job - e.job_begin;
  const long long row = local / per_row;
  const int kb = static_cast<int>(local - row * per_row);
  const size_t off = static_cast<size_t>(row) * n + kb * kRowBlock + 4 * lane;
  const uint2 xr = *reinterpret_cast<const uint2*>(e.x + off);
  const __half2 x01 = *reinterpret_cast<const __half2*>(&xr.x);
  const __half2 x23 = *reinterpret_cast<const __half2*>(&xr.y);
  float v[4] = {__low2float(x01), __high2float(x01), __low2float(x23), __high2float(x23)};
  if (e.s_in != nullptr) {
    const uint2 sr = *reinterpret_cast<const uint2*>(e.s_in + kb * kRowBlock + 4 * lane);
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
  const float factor = e.factor;
  uint4 o;
  o.x = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[0] * factor))) * 0x10001u;
  o.y = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[1] * factor))) * 0x10001u;
  o.z = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[2] * factor))) * 0x10001u;
  o.w = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[3] * factor))) * 0x10001u;
  *reinterpret_cast<uint4*>(e.xd + off) = o;
}

// Output transform of the layer kernels, for a group of layers: one warp per
// (layer, batch row, 128-row block): y = binary16(Hb(s_out (.) (scale (.)
// zacc))) and zacc := 0.  Launched as a programmatic dependent of the layer
// kernel; waits for it before reading.
__global__ void __launch_bounds__(kSmallThreads, 16) epi_kernel(const EpiGroup g) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long job = static_cast<long long>(blockIdx.x) * (kSmallThreads / 32) + (threadIdx.x >> 5);
  if (job >= g.jobs) return;
  int li = 0;
  {
    int hi = g.count - 1;  // the last layer whose first job is <= job
    while (li < hi) {
      const int mid = (li + hi + 1) >> 1;
      if (job >= g.e[mid].job_begin) li = mid; else hi = mid - 1;
    }
  }
  const EpiEntry& e = g.e[li];
  const int m = e.m;
  const int per_row = m / kRowBlock;
  const long long local = job - e.job_begin;
  const long long b = local / per_row;
  const int rb = static_cast<int>(local - b * per_row);
  const int r0 = rb * kRowBlock + 4 * lane;
  float4* zp = reinterpret_cast<float4*>(e.zacc + b * m + r0);
  const float4 z = __ldcg(zp);
  *zp = make_float4(0.f, 0.f, 0.f, 0.f);
  float v[4] = {z.x, z.y, z.z, z.w};
  {
    const uint2 sr = *reinterpret_cast<const uint2*>(e.scales + r0);
    const __half2 s01 = *reinterpret_cast<const __half2*>(&sr.x);
    const __half2 s23 = *reinterpret_cast<const __half2*>(&sr.y);
    v[0] *= __low2float(s01);
    v[1] *= __high2float(s01);
    v[2] *= __low2float(s23);
    v[3] *= __high2float(s23);
  }
  if (e.s_out != nullptr) {
    const uint2 sr = *reinterpret_cast<const uint2*>(e.s_out + r0);
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
  *reinterpret_cast<uint2*>(e.y + b * m + r0) = o;
}

template <int K, int CB>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const uint32_t* __restrict__ codes, int m, int n, __half* __restrict__ w) {
  const long long gid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  const int tiles_per_row = n / 16;
  const long long tiles = static_cast<long long>(m / 16) * tiles_per_row;
  if (gid >= tiles * 8) return;
  const long long tile = gid >> 3;
  const int p = static_cast<int>(gid & 7);
  const long long I = tile / tiles_per_row;
  const int J = static_cast<int>(tile - I * tiles_per_row);
  uint32_t wr[RowPair<K>::kPairWords];
  load_row_pair<K>(codes + tile * RowPair<K>::kTileWords, p, wr);
  uint32_t st[32];
  pair_states<K>(wr, st);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    uint32_t packed[8];
#pragma unroll
    for (int c = 0; c < 16; c += 2) packed[c / 2] = decode_pair<CB>(st[16 * k + c], st[16 * k + c + 1]);
    __half* dst = w + (I * 16 + 2 * p + k) * static_cast<long long>(n) + J * 16;
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  }
}

// The same decode, written as the dense tensor-core kernel's operand A: for
// every 128-row block rb and 64-column stage ks, a 16 KB image at byte
// (rb * (n / 64) + ks) * 16384 in the canonical K-major no-swizzle layout of a
// 128 x 64 binary16 operand: element (r, k) at byte
// ((k / 8) * 16 + r / 8) * 128 + (r % 8) * 16 + (k % 8) * 2.
// A warp decodes the four tiles of one stage in one tile row (16 rows x 64
// columns), whose image is eight 256-byte runs (one per 8-column group); the
// lanes' 16-byte row pieces are regrouped through shared memory so that each
// store instruction writes two whole runs.
template <int K, int CB>
__global__ void __launch_bounds__(kThreads)
    decode_aimg_kernel(const uint32_t* __restrict__ codes, int m, int n, unsigned char* __restrict__ aimg) {
  __shared__ uint4 runs[kThreads / 32][128];
  const long long gid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  const int tiles_per_row = n / 16;
  const long long tiles = static_cast<long long>(m / 16) * tiles_per_row;
  if (gid >= tiles * 8) return;  // whole warps: the tile count is a multiple of 8
  const int lane = threadIdx.x & 31;
  uint4* run = runs[threadIdx.x >> 5];
  const long long tile = gid >> 3;
  const int p = static_cast<int>(gid & 7);
  const long long I = tile / tiles_per_row;
  const int J = static_cast<int>(tile - I * tiles_per_row);
  uint32_t wr[RowPair<K>::kPairWords];
  load_row_pair<K>(codes + tile * RowPair<K>::kTileWords, p, wr);
  uint32_t st[32];
  pair_states<K>(wr, st);
  const int jt = J % 4;  // this lane's tile within the stage: 8-column groups 2 jt, 2 jt + 1
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    uint32_t packed[8];
#pragma unroll
    for (int c = 0; c < 16; c += 2) packed[c / 2] = decode_pair<CB>(st[16 * k + c], st[16 * k + c + 1]);
    const int r = 2 * p + k;  // row within the tile
    // run kg holds rows r of the tile row at (r / 8) * 8 + r % 8, 16 bytes each
    run[(2 * jt) * 16 + r] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    run[(2 * jt + 1) * 16 + r] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  }
  __syncwarp();
  // run kg goes to ((kg * 16) + 2 * (I % 8)) * 128 of the stage image: core
  // matrices r / 8 = 0, 1 of the tile row's two 8-row groups, contiguous
  unsigned char* stage = aimg + ((I / 8) * (n / 64) + J / 4) * 16384 + (I % 8) * 256;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int kg = 2 * i + (lane >> 4);
    const int off = lane & 15;
    *reinterpret_cast<uint4*>(stage + kg * 2048 + off * 16) = run[kg * 16 + off];
  }
}

template <int K>
exl3_status launch_decode_aimg_k(const uint32_t* codes, int codebook, int m, int n, unsigned char* aimg,
                                 cudaStream_t stream) {
  const long long threads = static_cast<long long>(m / 16) * (n / 16) * 8;
  const unsigned grid = static_cast<unsigned>((threads + kThreads - 1) / kThreads);
  switch (codebook) {
    case kCb3Inst: decode_aimg_kernel<K, kCb3Inst><<<grid, kThreads, 0, stream>>>(codes, m, n, aimg); break;
    case kCb1Mad: decode_aimg_kernel<K, kCb1Mad><<<grid, kThreads, 0, stream>>>(codes, m, n, aimg); break;
    case kCbMcg: decode_aimg_kernel<K, kCbMcg><<<grid, kThreads, 0, stream>>>(codes, m, n, aimg); break;
    default: decode_aimg_kernel<K, kCbMul1><<<grid, kThreads, 0, stream>>>(codes, m, n, aimg); break;
  }
  return launch_status();
}

template <int K>
exl3_status launch_decode_k(const uint32_t* codes, int codebook, int m, int n, __half* w,
                            cudaStream_t stream) {
  const long long threads = static_cast<long long>(m / 16) * (n / 16) * 8;
  const unsigned grid = static_cast<unsigned>((threads + kThreads - 1) / kThreads);
  switch (codebook) {
    case kCb3Inst: decode_kernel<K, kCb3Inst><<<grid, kThreads, 0, stream>>>(codes, m, n, w); break;
    case kCb1Mad: decode_kernel<K, kCb1Mad><<<grid, kThreads, 0, stream>>>(codes, m, n, w); break;
    case kCbMcg: decode_kernel<K, kCbMcg><<<grid, kThreads, 0, stream>>>(codes, m, n, w); break;
    default: decode_kernel<K, kCbMul1><<<grid, kThreads, 0, stream>>>(codes, m, n, w); break;
  }
  return launch_status();
}

}  // namespace

exl3_status launch_rht(const __half* in, const __half* signs, __half* out, int rows, int d,
                       cudaStream_t stream) {
  const long long blocks = static_cast<long long>(rows) * (d / kRowBlock);
  const long long per_cta = kThreads / 32;
  const unsigned grid = static_cast<unsigned>((blocks + per_cta - 1) / per_cta);
  rht_kernel<<<grid, kThreads, 0, stream>>>(in, signs, out, blocks, d);
  return launch_status();
}

exl3_status launch_bimg(const __half* x, const __half* s_in, __half* bimg, float* bsum, int M,
                        int nb, int n, cudaStream_t stream) {
  if (nb < 128) {
    BimgGroup g{};
    g.count = 1;
    g.e[0] = BimgEntry{x, s_in, bimg, bsum, n, 0};
    return launch_bimg_group(g, M, nb, stream);
  }
  constexpr int R = 8;
  const long long blocks = static_cast<long long>((M + nb - 1) / nb) * (nb / R) * (n / kRowBlock);
  const long long per_cta = kSmallThreads / 32;
  const unsigned grid = static_cast<unsigned>((blocks + per_cta - 1) / per_cta);
  bimg8_kernel<<<grid, kSmallThreads, 0, stream>>>(x, s_in, bimg, bsum, M, nb, n);
  return launch_status();
}

namespace {

template <typename G, typename Kern>
exl3_status launch_pdl_small(Kern kernel, const G& g, cudaStream_t stream) {
  const long long per_cta = kSmallThreads / 32;
  const unsigned grid = static_cast<unsigned>((g.jobs + per_cta - 1) / per_cta);
  if (grid == 0) return EXL3_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, g) != cudaSuccess) return EXL3_ERR_CUDA;
  return launch_status();
}

}  // namespace

float code_x_factor(int codebook) {
  return codebook == kCb1Mad ? x_factor<kCb1Mad>() : codebook == kCbMul1 ? x_factor<kCbMul1>() : 1.0f;
}

exl3_status launch_xdup_group(XdupGroup g, int codebook, cudaStream_t stream) {
  if (codebook >= 0)
    for (int i = 0; i < g.count; ++i) g.e[i].factor = code_x_factor(codebook);
  g.jobs = 0;
  for (int i = 0; i < g.count; ++i) {
    g.e[i].job_begin = g.jobs;
    g.jobs += static_cast<long long>(g.rows) * (g.e[i].n / kRowBlock);
  }
  return launch_pdl_small(xdup_kernel, g, stream);
}

exl3_status launch_epi_group(EpiGroup g, cudaStream_t stream) {
  g.jobs = 0;
  for (int i = 0; i < g.count; ++i) {
    g.e[i].job_begin = g.jobs;
    g.jobs += static_cast<long long>(g.rows) * (g.e[i].m / kRowBlock);
  }
  return launch_pdl_small(epi_kernel, g, stream);
}

exl3_status launch_bimg_group(BimgGroup g, int M, int nb, cudaStream_t stream) {
  if (nb >= 128) return EXL3_ERR_BATCH;  // wide tiles: launch_bimg
  g.M = M;
  g.nb = nb;
  g.jobs = 0;
  const long long rows = static_cast<long long>((M + nb - 1) / nb) * nb;
  for (int i = 0; i < g.count; ++i) {
    g.e[i].job_begin = g.jobs;
    g.jobs += rows * (g.e[i].n / kRowBlock);
  }
  return launch_pdl_small(bimg_kernel, g, stream);
}

exl3_status launch_xdup(const __half* x, const __half* s_in, uint32_t* xd, int rows, int n,
                        int codebook, cudaStream_t stream) {
  XdupGroup g{};
  g.count = 1;
  g.rows = rows;
  g.e[0].x = x;
  g.e[0].s_in = s_in;
  g.e[0].xd = xd;
  g.e[0].n = n;
  return launch_xdup_group(g, codebook, stream);
}

exl3_status launch_epi(float* zacc, const __half* scales, const __half* s_out, __half* y, int rows,
                       int m, cudaStream_t stream) {
  EpiGroup g{};
  g.count = 1;
  g.rows = rows;
  g.e[0].zacc = zacc;
  g.e[0].scales = scales;
  g.e[0].s_out = s_out;
  g.e[0].y = y;
  g.e[0].m = m;
  return launch_epi_group(g, stream);
}

exl3_status launch_decode_aimg(const uint32_t* codes, int K, int codebook, int m, int n,
                               unsigned char* aimg, cudaStream_t stream) {
  switch (K) {
    case 1: return launch_decode_aimg_k<1>(codes, codebook, m, n, aimg, stream);
    case 2: return launch_decode_aimg_k<2>(codes, codebook, m, n, aimg, stream);
    case 3: return launch_decode_aimg_k<3>(codes, codebook, m, n, aimg, stream);
    case 4: return launch_decode_aimg_k<4>(codes, codebook, m, n, aimg, stream);
    case 5: return launch_decode_aimg_k<5>(codes, codebook, m, n, aimg, stream);
    case 6: return launch_decode_aimg_k<6>(codes, codebook, m, n, aimg, stream);
    case 7: return launch_decode_aimg_k<7>(codes, codebook, m, n, aimg, stream);
    case 8: return launch_decode_aimg_k<8>(codes, codebook, m, n, aimg, stream);
    default: return EXL3_ERR_K;
  }
}

exl3_status launch_decode(const uint32_t* codes, int K, int codebook, int m, int n, __half* w,
                          cudaStream_t stream) {
  switch (K) {
    case 1: return launch_decode_k<1>(codes, codebook, m, n, w, stream);
    case 2: return launch_decode_k<2>(codes, codebook, m, n, w, stream);
    case 3: return launch_decode_k<3>(codes, codebook, m, n, w, stream);
    case 4: return launch_decode_k<4>(codes, codebook, m, n, w, stream);
    case 5: return launch_decode_k<5>(codes, codebook, m, n, w, stream);
    case 6: return launch_decode_k<6>(codes, codebook, m, n, w, stream);
    case 7: return launch_decode_k<7>(codes, codebook, m, n, w, stream);
    case 8: return launch_decode_k<8>(codes, codebook, m, n, w, stream);
    default: return EXL3_ERR_K;
  }
}

}  // namespace exl3
