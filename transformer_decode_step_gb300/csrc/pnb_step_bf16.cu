// pnb_step_bf16.cu - persistent step kernels for bf16 weights and KV cache.
#include "pnb_step_launch.cuh"

namespace pnb {
cudaError_t step_bf16(int hd, int G, const StepArgs &a, int grid, int smem, cudaStream_t st,
                      bool prepare, int *bps) {
  return step_dispatch<__nv_bfloat16>(hd, G, a, grid, smem, st, prepare, bps);
}
}  // namespace pnb
