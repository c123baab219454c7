// Host launchers of the dense prefill kernel (exl3_dense.cuh): operand A from
// images for every tile width, and the per-K dispatch of the fused variant.
#include "exl3_dense.cuh"

namespace exl3 {

int choose_dense_split(int units, int nstage, int grid) {
  // Splitting only the last partial round after whole rounds (224 units on
  // 152 SMs: 72 units in two K ranges) measured no faster: the partial sums'
  // reductions and the second pass cost what the idle SMs would have.  So
  // split only when there are fewer units than SMs.
  if (units >= grid) return 1;
  const int rem = units;
  int s = grid / rem;
  if (s > nstage / 16) s = nstage / 16;
  if (s > 16) s = 16;
  return s < 1 ? 1 : s;
}

int choose_fused_split(int units, int nstage, int grid, int rows) {
  // The fused kernel's stages cost several times those of the kernel on
  // decoded images, so a K split that evens out the rounds can pay for its
  // partial sums: minimise rounds x stages per item, charging each round of
  // split items for its reduction and fix-up, 3 + rows/64 stages (fitted on
  // the llama shapes at 48, 128 and 256 rows).
  if (units >= grid) return 1;
  const int charge = 3 + rows / 64;
  int best = 1;
  long long best_cost = nstage;
  for (int s = 2; s <= 16 && nstage / s >= 4; ++s) {
    const long long rounds = (static_cast<long long>(units) * s + grid - 1) / grid;
    const long long cost = rounds * ((nstage + s - 1) / s) + rounds * charge;
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

exl3_status launch_dense(const unsigned char* aimg, const __half* bimg, const __half* scales,
                         const __half* s_out, __half* y, float* zacc, uint32_t* cnt, int m, int n, int M,
                         int nb, int split, uint32_t* status, int debug_stall, cudaStream_t stream) {
  using namespace dense;
  if (split < 1 || split > n / kStageK) return EXL3_ERR_SHAPE;
  DenseParams p;
  p.aimg = aimg;
  p.bimg = bimg;
  p.scales = scales;
  p.s_out = s_out;
  p.y = y;
  p.zacc = zacc;
  p.cnt = cnt;
  p.status = status;
  p.m = m;
  p.n = n;
  p.M = M;
  p.debug_stall = debug_stall;
  p.codes = nullptr;
  p.zscale = 1.0f;
  switch (nb) {
    case 64:
      return launch_dense_kernel<64, 0, 0>(p, split, stream);
    case 128:
      return launch_dense_kernel<128, 0, 0>(p, split, stream);
    case 256:
      return launch_dense_kernel<256, 0, 0>(p, split, stream);
    default:
      return EXL3_ERR_SHAPE;
  }
}

exl3_status launch_fused(const uint32_t* codes, int K, int codebook, const __half* bimg, const __half* scales,
                         const __half* s_out, __half* y, float* zacc, uint32_t* cnt, int m, int n, int M,
                         int nb, int split, uint32_t* status, int debug_stall, cudaStream_t stream) {
  using namespace dense;
  if (split < 1 || split > n / kStageK) return EXL3_ERR_SHAPE;
  DenseParams p;
  p.aimg = nullptr;
  p.codes = codes;
  p.bimg = bimg;
  p.scales = scales;
  p.s_out = s_out;
  p.y = y;
  p.zacc = zacc;
  p.cnt = cnt;
  p.status = status;
  p.m = m;
  p.n = n;
  p.M = M;
  p.debug_stall = debug_stall;
  p.zscale = codebook == kCb1Mad ? x_factor<kCb1Mad>() : codebook == kCbMul1 ? x_factor<kCbMul1>() : 1.0f;
  switch (K) {
    case 1: return launch_fused_k1(p, codebook, nb, split, stream);
    case 2: return launch_fused_k2(p, codebook, nb, split, stream);
    case 3: return launch_fused_k3(p, codebook, nb, split, stream);
    case 4: return launch_fused_k4(p, codebook, nb, split, stream);
    case 5: return launch_fused_k5(p, codebook, nb, split, stream);
    case 6: return launch_fused_k6(p, codebook, nb, split, stream);
    case 7: return launch_fused_k7(p, codebook, nb, split, stream);
    case 8: return launch_fused_k8(p, codebook, nb, split, stream);
    default: return EXL3_ERR_K;
  }
}

}  // namespace exl3
