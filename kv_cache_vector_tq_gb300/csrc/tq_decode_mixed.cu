// Decode kernels instantiated for K and V caches at b + 1/2 bits per
// coordinate (b = 1..3: 1.5, 2.5 or 3.5 bits), 1, 2, 4 or 8 query heads per
// KV head.
#include "tq_decode_kernel.cuh"

namespace tq {

namespace {

template <int B>
cudaError_t mixed_g(const StepParams& p, int G, int groups, cudaStream_t st) {
  switch (G) {
    case 1: return run_step<B, B, 1, false, true>(p, groups, st);
    case 2: return run_step<B, B, 2, false, true>(p, groups, st);
    case 4: return run_step<B, B, 4, false, true>(p, groups, st);
    case 8: return run_step<B, B, 8, false, true>(p, groups, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_run_mixed(const StepParams& p, int b, int G, int groups, cudaStream_t st) {
  switch (b) {
    case 1: return mixed_g<1>(p, G, groups, st);
    case 2: return mixed_g<2>(p, G, groups, st);
    case 3: return mixed_g<3>(p, G, groups, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
