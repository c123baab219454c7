// exl3_gemv_noalloc: the batch-1 fused layer for callers that cannot allocate
// device memory.
//
// exl3_gemv needs a caller-provided workspace (fp32 row sums and counters).  Some callers cannot provide one: code that
// runs where cudaMalloc is unavailable or forbidden (inside a host callback or
// a custom allocator's own hooks, a plugin whose host framework owns every
// allocation, a real-time loop that must never allocate).  This entry point
// takes the same inputs and output but keeps its scratch in a fixed,
// file-scope device array instead, so it allocates nothing.
//
// The array (EXL3_NOALLOC_SCRATCH_BYTES) lives on every GPU that loads the
// library until the process exits.  All calls share it, so calls whose kernels
// can overlap on the GPU (different streams, or different host threads on one
// device) race and must be serialized by the caller.
#include <cuda_runtime.h>

#include <atomic>

#include "exl3_host.cuh"

namespace exl3 {
namespace {

constexpr size_t kScratchBytes = EXL3_NOALLOC_SCRATCH_BYTES;

// The shared scratch.  In host code this name is only a handle for the runtime;
// the kernels get the device address obtained below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
// Per device, the array's device address once looked up.  Host threads may
// make their first calls on a device at the same time: each may look the
// address up (the runtime returns the same value) and the stores and loads are
// atomic, so no thread reads a half-written pointer.
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch on device `dev` (which must be current),
// looked up once and cached.
exl3_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return EXL3_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return EXL3_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return EXL3_OK;
}

}  // namespace
}  // namespace exl3

using namespace exl3;

extern "C" exl3_status exl3_gemv_noalloc(const uint32_t* codes, int K, int codebook, int m, int n,
                                         const exl3_half* s_in, const exl3_half* s_out,
                                         const exl3_half* scales, const exl3_half* x,
                                         exl3_half* y, exl3_stream_t stream) {
  exl3_status st = check_shape(m, n);
  if (st != EXL3_OK) return st;
  if ((st = check_k_cb(K, codebook)) != EXL3_OK) return st;
  if (!codes || !scales || !x || !y) return EXL3_ERR_NULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(y) ||
      (s_in && !aligned16(s_in)) || (s_out && !aligned16(s_out)))
    return EXL3_ERR_ALIGN;

  // Scratch layout as in the workspace of exl3_gemv at batch 1: the block
  // counters and the status word, the m fp32 row sums, then the n 32-bit x
  // pairs of the warp-shuffle kernel.
  const size_t zero_bytes = bimg_offset(m, 1);  // counters, status word and row sums
  const size_t need = zero_bytes + align256(sizeof(uint32_t) * static_cast<size_t>(n));
  if (need > kScratchBytes) return EXL3_ERR_SCRATCH;

  // The array's address is per device: it must be the address on the device
  // that runs `stream`, which must be the current device.
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sdev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaStreamGetDevice(cs, &sdev) != cudaSuccess || sdev != dev)
    return EXL3_ERR_CUDA;
  void* scratch = nullptr;
  if ((st = scratch_address(dev, &scratch)) != EXL3_OK) return st;
  // The row sums must start at zero; the array keeps whatever the previous
  // call left, so clear them (and the counters) on the stream first.
  if (cudaMemsetAsync(scratch, 0, zero_bytes, cs) != cudaSuccess) return EXL3_ERR_CUDA;

  char* base = static_cast<char*>(scratch);
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
  return run_shuffle(a, 1, reinterpret_cast<float*>(base + zacc_offset(m)),
                     reinterpret_cast<uint32_t*>(base + zero_bytes), cs);
}
