// k_step_128.cu -- the persistent decode-step kernel for head_dim 128 (see k_step.cuh),
// and the dispatch over head dims.
#include "k_step.cuh"

namespace hfa {

cudaError_t launch_step_64(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                           int grid, cudaStream_t s);
cudaError_t launch_step_256(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, cudaStream_t s);
cudaError_t launch_step_512(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, cudaStream_t s);

cudaError_t launch_step(const StepArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int hd,
                        int grid, cudaStream_t s) {
  if (hd == 64) return launch_step_64(a, tk, tv, grid, s);
  if (hd == 128) return step::launch_step_hd<128>(a, tk, tv, grid, s);
  if (hd == 512) return launch_step_512(a, tk, tv, grid, s);
  return launch_step_256(a, tk, tv, grid, s);
}

int step_keys_per_tile(int hd) {
  return hd == 64    ? step::Attn<64>::T
         : hd == 128 ? step::Attn<128>::T
         : hd == 256 ? step::Attn<256>::T
                     : step::Attn<512>::T;
}

size_t step_smem_bytes() { return step::kSmem; }
size_t step_stage_bytes() { return step::kStageBytes; }
int step_threads() { return step::kThreads; }
int step_batch_tiles(int batch) { return batch <= 4 ? 1 : (batch <= 8 ? 2 : 4); }

}  // namespace hfa
