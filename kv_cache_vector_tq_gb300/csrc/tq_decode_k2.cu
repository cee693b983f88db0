// Decode kernels instantiated for key codes of 2 bits (every value width and
// GQA; one translation unit per key width so that they compile in parallel).
#include "tq_decode_kernel.cuh"

namespace tq {

cudaError_t decode_run_k2(const StepParams& p, int bv, int G, int groups, cudaStream_t st) {
  return run_step_v<2>(p, bv, G, groups, st);
}

}  // namespace tq
