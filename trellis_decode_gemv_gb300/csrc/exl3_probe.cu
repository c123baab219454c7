// exl3_probe_int: the integer-throughput probe behind the INT32 term of the
// layer roofline ("Trellis Quantization" Part three counts the decode's cost in
// integer instructions per weight against the GPU's integer issue rate).
//
// Every thread runs kChains = 8 independent dependency chains of one
// instruction kind (or an even mix of kinds), 4 * iters instructions each, so
// the pipes see as many independent instructions as they can take and latency
// does not bind.  The caller times the launch on its stream; ops = blocks *
// 256 threads * 8 chains * 4 * iters.  The chains' results go to out[blocks *
// 256] so that nothing is optimised away.
#include <cuda_runtime.h>

#include "exl3_host.cuh"

namespace exl3 {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kChains = 8;

template <int KIND>
__device__ __forceinline__ void probe_op(uint32_t& x, uint32_t y, uint32_t a, uint32_t b, int c) {
  // KIND 5 and 6 interleave kinds over the chains (independent chains of
  // different kinds, in equal numbers).
  constexpr int kinds5[2] = {0, 1};
  constexpr int kinds6[4] = {0, 3, 1, 2};
  const int k = KIND == 5 ? kinds5[c & 1] : KIND == 6 ? kinds6[c & 3] : KIND;
  if (k == 0) asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(x) : "r"(a), "r"(b));
  if (k == 1) asm volatile("lop3.b32 %0, %0, %1, %2, 0x6A;" : "+r"(x) : "r"(y), "r"(b));
  if (k == 2) asm volatile("shf.l.wrap.b32 %0, %0, %1, 5;" : "+r"(x) : "r"(y));
  if (k == 3) asm volatile("dp4a.u32.u32 %0, %0, %1, %2;" : "+r"(x) : "r"(a), "r"(b));
  if (k == 4) asm volatile("prmt.b32 %0, %0, %1, 0x5410;" : "+r"(x) : "r"(y));
}

template <int KIND>
__global__ void __launch_bounds__(kProbeThreads) probe_kernel(uint32_t* __restrict__ out, int iters) {
  uint32_t x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) x[c] = threadIdx.x * 2654435761u + blockIdx.x + 977u * c;
  const uint32_t a = 0x9E3779B9u, b = 0x7F4A7C15u;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
#pragma unroll
      for (int c = 0; c < kChains; ++c) probe_op<KIND>(x[c], x[(c + 1) % kChains], a, b, c);
    }
  }
  uint32_t v = 0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) v ^= x[c];
  out[static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x] = v;
}

}  // namespace
}  // namespace exl3

using namespace exl3;

extern "C" exl3_status exl3_probe_int(int kind, uint32_t* out, int blocks, int iters, exl3_stream_t stream) {
  if (kind < 0 || kind > 6) return EXL3_ERR_BATCH;
  if (blocks < 1 || iters < 1) return EXL3_ERR_SHAPE;
  if (out == nullptr) return EXL3_ERR_NULL;
  if (!aligned16(out)) return EXL3_ERR_ALIGN;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int rounds = iters;
  switch (kind) {
    case 0: probe_kernel<0><<<blocks, kProbeThreads, 0, cs>>>(out, rounds); break;
    case 1: probe_kernel<1><<<blocks, kProbeThreads, 0, cs>>>(out, rounds); break;
    case 2: probe_kernel<2><<<blocks, kProbeThreads, 0, cs>>>(out, rounds); break;
    case 3: probe_kernel<3><<<blocks, kProbeThreads, 0, cs>>>(out, rounds); break;
    case 4: probe_kernel<4><<<blocks, kProbeThreads, 0, cs>>>(out, rounds); break;
    case 5: probe_kernel<5><<<blocks, kProbeThreads, 0, cs>>>(out, rounds); break;
    default: probe_kernel<6><<<blocks, kProbeThreads, 0, cs>>>(out, rounds); break;
  }
  return launch_status();
}
