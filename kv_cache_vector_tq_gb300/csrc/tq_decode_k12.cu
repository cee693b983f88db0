// Decode kernels instantiated for key codes of 1 and 2 bits.
#include "tq_decode_kernel.cuh"

namespace tq {

cudaError_t decode_run_k12(const StepParams& p, int bk, int bv, int G, int groups, cudaStream_t st) {
  return bk == 1 ? run_step_v<1>(p, bv, G, groups, st) : run_step_v<2>(p, bv, G, groups, st);
}

}  // namespace tq
