// pnb_step_launch.cuh - cooperative launch of the persistent step kernel for
// one (storage type, head_dim) pair, dispatching on the query-head group size.
#pragma once

#include "pnb_step.cuh"

namespace pnb {

template <typename T, int HD, int G>
cudaError_t step_launch_one(const StepArgs &a, int grid, int smem, cudaStream_t st, bool prepare,
                            int *blocks_per_sm) {
  auto kern = k_step<T, HD, G>;
  if (prepare) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kern, kStepThreads, smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStepThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int HD>
cudaError_t step_dispatch_g(int G, const StepArgs &a, int grid, int smem, cudaStream_t st, bool prepare,
                            int *bps) {
  switch (G) {
    case 1: return step_launch_one<T, HD, 1>(a, grid, smem, st, prepare, bps);
    case 2: return step_launch_one<T, HD, 2>(a, grid, smem, st, prepare, bps);
    case 4: return step_launch_one<T, HD, 4>(a, grid, smem, st, prepare, bps);
    case 8:
      if constexpr (HD <= 64) return step_launch_one<T, HD, 8>(a, grid, smem, st, prepare, bps);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t step_dispatch(int hd, int G, const StepArgs &a, int grid, int smem, cudaStream_t st,
                          bool prepare, int *bps) {
  switch (hd) {
    case 32: return step_dispatch_g<T, 32>(G, a, grid, smem, st, prepare, bps);
    case 64: return step_dispatch_g<T, 64>(G, a, grid, smem, st, prepare, bps);
    case 128: return step_dispatch_g<T, 128>(G, a, grid, smem, st, prepare, bps);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pnb
