// pnb_step_f32.cu - persistent step kernels for fp32 weights and KV cache.
#include "pnb_step_launch.cuh"

namespace pnb {
cudaError_t step_f32(int hd, int G, const StepArgs &a, int grid, int smem, cudaStream_t st,
                     bool prepare, int *bps) {
  return step_dispatch<float>(hd, G, a, grid, smem, st, prepare, bps);
}
}  // namespace pnb
