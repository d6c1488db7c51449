// k_step_64.cu -- the persistent decode-step kernel for head_dim 64 (see k_step.cuh).
#include "k_step.cuh"

namespace hfa {

cudaError_t launch_step_64(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                           int grid, cudaStream_t s) {
  return step::launch_step_hd<64>(a, tk, tv, grid, s);
}

}  // namespace hfa
