// Decode kernels instantiated for key codes of 3 and 4 bits.
#include "tq_decode_kernel.cuh"

namespace tq {

cudaError_t decode_run_k34(const StepParams& p, int bk, int bv, int G, int groups, cudaStream_t st) {
  return bk == 3 ? run_step_v<3>(p, bv, G, groups, st) : run_step_v<4>(p, bv, G, groups, st);
}

}  // namespace tq
