// Tail-biting Viterbi encoder of the bitshift trellis on the GPU ("Trellis
// Quantization" Part seven: the Viterbi search keeps, for every state, the
// cheapest path that ends in it and reads the best path back at the end; Part
// eight: the L = 16-bit window moving K bits per step, so the predecessors of
// state s' are h * 2^(16-K) + (s' >> K), and the two-pass tail-biting
// approximation: run on the sequence rotated by half its length, take the
// state in the middle, run again on the original sequence starting from that
// state with the appended bits that wrap past the end of the stream forced to
// repeat its first bits).
//
// One CTA per tile (256 steps), persistent over tiles.  The search carries,
// per group g = s' >> K, best(g) = min over the 2^K predecessors of their path
// cost: 2^(16-K) binary32 values in shared memory (128 KB at K = 1), updated
// in place between two barriers per step.  Each path cost is
// best(s >> K) + (v(s) - x_t)^2 evaluated as three binary32 roundings in that
// order; the smallest predecessor index wins ties, and at the end the
// smallest state.  v(s) is the code's binary16 value, cached for all 2^16
// states in shared memory for K >= 2 and computed in place for K = 1.  The
// predecessor choices (one byte per group and step) go to a per-CTA slot of
// the workspace, from which thread 0 reads the path back.
#include "exl3_device.cuh"
#include "exl3_host.cuh"

namespace exl3 {
namespace enc {

constexpr int kThreads = 1024;
constexpr int kSteps = 256;
constexpr int kStates = 1 << 16;

template <int K>
struct Cfg {
  static constexpr int kNb = 1 << K;
  static constexpr int kLow = 1 << (16 - K);         // groups
  static constexpr int kQStride = 1 << (16 - 2 * K);  // (h * kLow + g) >> K = h * kQStride + (g >> K)
  static constexpr int kPer = kLow >= kThreads ? kLow / kThreads : 1;
  static constexpr bool kCache = K >= 2;
  static constexpr size_t kBestBytes = sizeof(float) * kLow;
  static constexpr size_t kCacheBytes = kCache ? sizeof(__half) * kStates : 0;
  static constexpr size_t kSlotBytes = static_cast<size_t>(kSteps) * kLow;
};

struct EncShared {
  float x[kSteps];
  uint32_t states[kSteps];
  uint8_t fmask[kSteps];
  uint8_t fbits[kSteps];
  float red_c[kThreads / 32];
  uint32_t red_s[kThreads / 32];
  uint32_t s_star;
  uint32_t s_last;
  float cost;
};

struct EncParams {
  const float* target;
  uint32_t* words;
  float* cost;
  uint8_t* back;
  int tiles;
};

template <int K, int CB>
__device__ __forceinline__ float value_of(const __half* vcache, uint32_t s) {
  if constexpr (Cfg<K>::kCache) {
    return __half2float(vcache[s]);
  } else {
    return __half2float(decode_state<CB>(s));
  }
}

// Minimum over the 2^K predecessors of one group g at one step: the path
// costs best(h * kQStride + (g >> K)) + (v(s) - x)^2, s = h * kLow + g, with the
// appended bits of s checked against (fm, fb) when Forced.
template <int K, int CB, bool First, bool Forced>
__device__ __forceinline__ float group_min(const float* best, const __half* vcache, int g, float xp, int start,
                                           uint32_t fm, uint32_t fb, int& bh) {
  using C = Cfg<K>;
  const float inf = __int_as_float(0x7f800000);
  float bc = inf;
  bh = 0;
#pragma unroll 4
  for (int h = 0; h < C::kNb; ++h) {
    const uint32_t s = static_cast<uint32_t>(h) * C::kLow + g;
    float base;
    if constexpr (First)
      base = (start < 0 || s == static_cast<uint32_t>(start)) ? 0.0f : inf;
    else
      base = best[h * C::kQStride + (g >> K)];
    const float d = __fsub_rn(value_of<K, CB>(vcache, s), xp);
    float c = __fadd_rn(base, __fmul_rn(d, d));
    if constexpr (Forced) {
      if ((s & fm) != fb) c = inf;
    }
    if (c < bc) {
      bc = c;
      bh = h;
    }
  }
  return bc;
}

// Small K: one thread takes a whole butterfly q (the 2^K predecessor groups
// h * kQStride + q feed exactly the 2^K successor groups q * 2^K + b), so each
// predecessor minimum is read once for 2^K outputs and the values of the 2^K
// consecutive states h * kLow + q * 2^K + b come in one shared-memory load.
template <int K>
struct ByQ {
  static constexpr bool kOn = K <= 3;
  static constexpr int kQ = 1 << (16 - 2 * K);  // butterflies
  static constexpr int kPerThread = kQ >= kThreads ? kQ / kThreads : 1;
};

template <int K, int CB, bool First, bool Forced>
__device__ __forceinline__ void butterfly(const float* best, const __half* vcache, int q, float xp, int start,
                                          uint32_t fm, uint32_t fb, float (&oc)[1 << K], uint64_t& packed_bh) {
  using C = Cfg<K>;
  constexpr int NB = C::kNb;
  const float inf = __int_as_float(0x7f800000);
  int bh[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    oc[b] = inf;
    bh[b] = 0;
  }
#pragma unroll
  for (int h = 0; h < NB; ++h) {
    const uint32_t s0 = static_cast<uint32_t>(h) * C::kLow + static_cast<uint32_t>(q) * NB;
    float base = First ? 0.0f : best[h * C::kQStride + q];
    float v[NB];
    if constexpr (C::kCache && NB == 4) {
      const uint2 r = *reinterpret_cast<const uint2*>(vcache + s0);
      const __half2 a = *reinterpret_cast<const __half2*>(&r.x);
      const __half2 c = *reinterpret_cast<const __half2*>(&r.y);
      v[0] = __low2float(a);
      v[1] = __high2float(a);
      v[2] = __low2float(c);
      v[3] = __high2float(c);
    } else if constexpr (C::kCache && NB == 8) {
      const uint4 r = *reinterpret_cast<const uint4*>(vcache + s0);
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 a = *reinterpret_cast<const __half2*>(&w[i]);
        v[2 * i] = __low2float(a);
        v[2 * i + 1] = __high2float(a);
      }
    } else {
#pragma unroll
      for (int b = 0; b < NB; ++b) v[b] = value_of<K, CB>(vcache, s0 + b);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const uint32_t s = s0 + b;
      float bs = base;
      if constexpr (First) bs = (start < 0 || s == static_cast<uint32_t>(start)) ? 0.0f : inf;
      const float d = __fsub_rn(v[b], xp);
      float c = __fadd_rn(bs, __fmul_rn(d, d));
      if constexpr (Forced) {
        if ((s & fm) != fb) c = inf;
      }
      if (c < oc[b]) {
        oc[b] = c;
        bh[b] = h;
      }
    }
  }
  static_assert(NB <= 8, "one byte per choice, at most eight in 64 bits");
  packed_bh = 0;
#pragma unroll
  for (int b = 0; b < NB; ++b) packed_bh |= static_cast<uint64_t>(bh[b]) << (8 * b);
}

// One Viterbi pass over the tile's 256 steps.  rotated: x_t = target[(t + 128)
// % 256]; start < 0: any first state; forced: the pass-two constraints in
// sh.fmask / sh.fbits.  Leaves the cheapest final state and its cost in
// sh.s_last / sh.cost.
template <int K, int CB>
__device__ void viterbi_pass(EncShared& sh, float* best, const __half* vcache, uint8_t* back, bool rotated,
                             int start, bool forced) {
  using C = Cfg<K>;
  const int tid = threadIdx.x;
  const float inf = __int_as_float(0x7f800000);
  for (int t = 1; t < kSteps; ++t) {
    const int tp = t - 1;  // the step whose path costs are minimised here
    const float xp = sh.x[rotated ? (tp + kSteps / 2) & (kSteps - 1) : tp];
    const uint32_t fm = forced ? sh.fmask[tp] : 0u;
    const uint32_t fb = forced ? sh.fbits[tp] : 0u;
    if constexpr (ByQ<K>::kOn) {
      constexpr int NB = C::kNb;
      float oc[ByQ<K>::kPerThread][NB];
#pragma unroll
      for (int j = 0; j < ByQ<K>::kPerThread; ++j) {
        const int q = tid + j * kThreads;
        uint64_t pk;
        if (tp == 0)
          butterfly<K, CB, true, false>(best, vcache, q, xp, start, fm, fb, oc[j], pk);
        else if (fm != 0u)
          butterfly<K, CB, false, true>(best, vcache, q, xp, start, fm, fb, oc[j], pk);
        else
          butterfly<K, CB, false, false>(best, vcache, q, xp, start, fm, fb, oc[j], pk);
        // the 2^K predecessor choices of groups q * 2^K .. + 2^K - 1, one byte each
        uint8_t* bp = back + static_cast<size_t>(t) * C::kLow + static_cast<size_t>(q) * NB;
        if constexpr (NB == 2) {
          *reinterpret_cast<uint16_t*>(bp) = static_cast<uint16_t>(pk);
        } else if constexpr (NB == 4) {
          *reinterpret_cast<uint32_t*>(bp) = static_cast<uint32_t>(pk);
        } else {
          *reinterpret_cast<uint64_t*>(bp) = pk;
        }
      }
      __syncthreads();  // every read of best for this step is done
#pragma unroll
      for (int j = 0; j < ByQ<K>::kPerThread; ++j) {
        const int q = tid + j * kThreads;
#pragma unroll
        for (int b = 0; b < NB; ++b) best[q * NB + b] = oc[j][b];
      }
      __syncthreads();
    } else {
    float out[C::kPer];
#pragma unroll
    for (int j = 0; j < C::kPer; ++j) {
      const int g = tid + j * kThreads;
      out[j] = inf;
      if (g < C::kLow) {
        int bh;
        // the first step and the forced steps (the last few of pass two) are
        // uniform branches; the common step checks nothing
        if (tp == 0)
          out[j] = group_min<K, CB, true, false>(best, vcache, g, xp, start, fm, fb, bh);
        else if (fm != 0u)
          out[j] = group_min<K, CB, false, true>(best, vcache, g, xp, start, fm, fb, bh);
        else
          out[j] = group_min<K, CB, false, false>(best, vcache, g, xp, start, fm, fb, bh);
        back[static_cast<size_t>(t) * C::kLow + g] = static_cast<uint8_t>(bh);
      }
    }
    __syncthreads();  // every read of best for this step is done
#pragma unroll
    for (int j = 0; j < C::kPer; ++j) {
      const int g = tid + j * kThreads;
      if (g < C::kLow) best[g] = out[j];
    }
    __syncthreads();
    }
  }
  // final step: cost of every state, the cheapest (smallest state on ties)
  {
    const int tp = kSteps - 1;
    const float xp = sh.x[rotated ? (tp + kSteps / 2) & (kSteps - 1) : tp];
    const uint32_t fm = forced ? sh.fmask[tp] : 0u;
    const uint32_t fb = forced ? sh.fbits[tp] : 0u;
    float bc = inf;
    uint32_t bs = 0xFFFFFFFFu;
    for (uint32_t s = tid; s < static_cast<uint32_t>(kStates); s += kThreads) {
      const float d = __fsub_rn(value_of<K, CB>(vcache, s), xp);
      float c = __fadd_rn(best[s >> K], __fmul_rn(d, d));
      if ((s & fm) != fb) c = inf;
      if (c < bc) {
        bc = c;
        bs = s;
      }
    }
    // warp then block reduction of (cost, state), lexicographic
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float oc = __shfl_xor_sync(0xFFFFFFFFu, bc, o);
      const uint32_t os = __shfl_xor_sync(0xFFFFFFFFu, bs, o);
      if (oc < bc || (oc == bc && os < bs)) {
        bc = oc;
        bs = os;
      }
    }
    const int lane = tid & 31;
    const int warp = tid >> 5;
    if (lane == 0) {
      sh.red_c[warp] = bc;
      sh.red_s[warp] = bs;
    }
    __syncthreads();
    if (tid == 0) {
      float c = sh.red_c[0];
      uint32_t s = sh.red_s[0];
      for (int w = 1; w < kThreads / 32; ++w)
        if (sh.red_c[w] < c || (sh.red_c[w] == c && sh.red_s[w] < s)) {
          c = sh.red_c[w];
          s = sh.red_s[w];
        }
      sh.s_last = s;
      sh.cost = c;
    }
    __syncthreads();
  }
}

template <int K, int CB>
__global__ void __launch_bounds__(kThreads, 1) encode_kernel(const EncParams p) {
  using C = Cfg<K>;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ EncShared sh;
  float* best = reinterpret_cast<float*>(smem);
  const __half* vcache = reinterpret_cast<const __half*>(smem + C::kBestBytes);
  const int tid = threadIdx.x;
  uint8_t* back = p.back + static_cast<size_t>(blockIdx.x) * C::kSlotBytes;

  if constexpr (C::kCache) {
    __half* vc = reinterpret_cast<__half*>(smem + C::kBestBytes);
    for (uint32_t s = tid; s < static_cast<uint32_t>(kStates); s += kThreads) vc[s] = decode_state<CB>(s);
  }

  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
    if (tid < kSteps) sh.x[tid] = p.target[static_cast<size_t>(tile) * kSteps + tid];
    __syncthreads();

    // pass one: the rotated sequence, free start; its middle state
    viterbi_pass<K, CB>(sh, best, vcache, back, true, -1, false);
    if (tid == 0) {
      uint32_t s = sh.s_last;
      for (int t = kSteps - 1; t > kSteps / 2; --t) {
        const uint32_t g = (s >> K) & (C::kLow - 1);
        s = g | ((static_cast<uint32_t>(back[static_cast<size_t>(t) * C::kLow + g]) & (C::kNb - 1)) << (16 - K));
      }
      sh.s_star = s;
    }
    __syncthreads();
    const uint32_t s_star = sh.s_star;
    // pass two's constraints: appended bits that lie past the end of the
    // circular stream repeat the stream's first bits, i.e. those of s_star
    if (tid < kSteps) {
      uint32_t mask = 0, bits = 0;
      if (tid >= 1) {
        const int first = K * (tid - 1) + 16;
        for (int i = 0; i < K; ++i) {
          const int j = first + i;
          if (j >= kSteps * K) {
            const int shift = K - 1 - i;
            mask |= 1u << shift;
            bits |= ((s_star >> (15 - (j - kSteps * K))) & 1u) << shift;
          }
        }
      }
      sh.fmask[tid] = static_cast<uint8_t>(mask);
      sh.fbits[tid] = static_cast<uint8_t>(bits);
    }
    __syncthreads();

    // pass two: the original sequence from s_star
    viterbi_pass<K, CB>(sh, best, vcache, back, false, static_cast<int>(s_star), true);
    if (tid == 0) {
      uint32_t s = sh.s_last;
      sh.states[kSteps - 1] = s;
      for (int t = kSteps - 1; t > 0; --t) {
        const uint32_t g = (s >> K) & (C::kLow - 1);
        s = g | ((static_cast<uint32_t>(back[static_cast<size_t>(t) * C::kLow + g]) & (C::kNb - 1)) << (16 - K));
        sh.states[t - 1] = s;
      }
      p.cost[tile] = sh.cost;
    }
    __syncthreads();
    // the stream: the first window, then the K bits appended at each step,
    // MSB first in 32-bit words
    if (tid < 8 * K) {
      uint32_t w = 0;
      for (int b = 0; b < 32; ++b) {
        const int j = 32 * tid + b;
        uint32_t bit;
        if (j < 16) {
          bit = (s_star >> (15 - j)) & 1u;
        } else {
          const int t = (j - 16) / K + 1;
          const int i = (j - 16) % K;
          bit = (sh.states[t] >> (K - 1 - i)) & 1u;
        }
        w |= bit << (31 - b);
      }
      p.words[static_cast<size_t>(tile) * 8 * K + tid] = w;
    }
    __syncthreads();
  }
}

template <int K, int CB>
exl3_status launch_encode_kc(const EncParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<K>;
  const size_t smem = C::kBestBytes + C::kCacheBytes;
  if (cudaFuncSetAttribute(encode_kernel<K, CB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return EXL3_ERR_CUDA;
  encode_kernel<K, CB><<<grid, kThreads, smem, stream>>>(p);
  return launch_status();
}

template <int K>
exl3_status launch_encode_k(const EncParams& p, int codebook, int grid, cudaStream_t stream) {
  switch (codebook) {
    case kCb3Inst: return launch_encode_kc<K, kCb3Inst>(p, grid, stream);
    case kCb1Mad: return launch_encode_kc<K, kCb1Mad>(p, grid, stream);
    case kCbMcg: return launch_encode_kc<K, kCbMcg>(p, grid, stream);
    default: return launch_encode_kc<K, kCbMul1>(p, grid, stream);
  }
}

inline size_t slot_bytes(int K) { return static_cast<size_t>(kSteps) << (16 - K); }

}  // namespace enc
}  // namespace exl3

using namespace exl3;

extern "C" size_t exl3_encode_workspace_bytes(int K, int ctas) {
  if (K < 1 || K > 8 || ctas < 1) return 0;
  return enc::slot_bytes(K) * static_cast<size_t>(ctas);
}

extern "C" exl3_status exl3_encode_tiles(const float* target, int tiles, int K, int codebook, uint32_t* words,
                                         float* cost, void* workspace, size_t workspace_bytes,
                                         exl3_stream_t stream) {
  if (tiles < 1) return EXL3_ERR_SHAPE;
  exl3_status st = check_k_cb(K, codebook);
  if (st != EXL3_OK) return st;
  if (!target || !words || !cost) return EXL3_ERR_NULL;
  if (!aligned16(target) || !aligned16(words)) return EXL3_ERR_ALIGN;
  if (!workspace || workspace_bytes < enc::slot_bytes(K)) return EXL3_ERR_WORKSPACE;
  const size_t slots = workspace_bytes / enc::slot_bytes(K);
  int grid = device_sm_count();
  if (static_cast<size_t>(grid) > slots) grid = static_cast<int>(slots);
  if (grid > tiles) grid = tiles;
  enc::EncParams p;
  p.target = target;
  p.words = words;
  p.cost = cost;
  p.back = static_cast<uint8_t*>(workspace);
  p.tiles = tiles;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  switch (K) {
    case 1: return enc::launch_encode_k<1>(p, codebook, grid, cs);
    case 2: return enc::launch_encode_k<2>(p, codebook, grid, cs);
    case 3: return enc::launch_encode_k<3>(p, codebook, grid, cs);
    case 4: return enc::launch_encode_k<4>(p, codebook, grid, cs);
    case 5: return enc::launch_encode_k<5>(p, codebook, grid, cs);
    case 6: return enc::launch_encode_k<6>(p, codebook, grid, cs);
    case 7: return enc::launch_encode_k<7>(p, codebook, grid, cs);
    default: return enc::launch_encode_k<8>(p, codebook, grid, cs);
  }
}
