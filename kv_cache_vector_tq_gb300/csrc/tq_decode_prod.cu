// Decode kernels instantiated for TurboQuant_Prod keys: (b−1)-bit MSE codes of
// 1 to 3 bits plus the QJL sign words, values of 1 to 4 bits, 1, 2 or 4 query
// heads per KV head.
#include "tq_decode_kernel.cuh"

namespace tq {

namespace {

template <int BK, int BV>
cudaError_t prod_g(const StepParams& p, int G, int groups, cudaStream_t st) {
  switch (G) {
    case 1: return run_step<BK, BV, 1, true>(p, groups, st);
    case 2: return run_step<BK, BV, 2, true>(p, groups, st);
    case 4: return run_step<BK, BV, 4, true>(p, groups, st);
  }
  return cudaErrorInvalidValue;
}

template <int BK>
cudaError_t prod_v(const StepParams& p, int bv, int G, int groups, cudaStream_t st) {
  switch (bv) {
    case 1: return prod_g<BK, 1>(p, G, groups, st);
    case 2: return prod_g<BK, 2>(p, G, groups, st);
    case 3: return prod_g<BK, 3>(p, G, groups, st);
    case 4: return prod_g<BK, 4>(p, G, groups, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_run_prod(const StepParams& p, int bk, int bv, int G, int groups, cudaStream_t st) {
  switch (bk) {
    case 1: return prod_v<1>(p, bv, G, groups, st);
    case 2: return prod_v<2>(p, bv, G, groups, st);
    case 3: return prod_v<3>(p, bv, G, groups, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
