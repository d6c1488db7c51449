// k_step_512.cu -- the persistent decode-step kernel for head_dim 512 (see k_step.cuh):
// the global layers of the model the pages describe (two KV heads of 512 dims).
#include "k_step.cuh"

namespace hfa {

cudaError_t launch_step_512(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, cudaStream_t s) {
  return step::launch_step_hd<512>(a, tk, tv, grid, s);
}

}  // namespace hfa
