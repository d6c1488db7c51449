// k_step_256.cu -- the persistent decode-step kernel for head_dim 256 (see k_step.cuh).
#include "k_step.cuh"

namespace hfa {

cudaError_t launch_step_256(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                           int grid, cudaStream_t s) {
  return step::launch_step_hd<256>(a, tk, tv, grid, s);
}

}  // namespace hfa
