// The interpreted variants of the fused-group kernels: the group's operator
// program runs on the register-stack machine (fg_device.cuh).  The compiled
// variants (jit.cpp) share the same pipeline (group_kernels.cuh).
#include <cuda_runtime.h>

#include "group_kernels.cuh"
#include "launch.h"

namespace fg {

template <int D, int S>
__global__ void __launch_bounds__(kThreads, D <= 4 ? 2 : 1) fg_ew_group_kernel(const __grid_constant__ GroupParams P) {
  ew_body<InterpProg<D, S>>(P);
}

template <int D, int S>
__global__ void __launch_bounds__(kThreads, D <= 4 ? 2 : 1)
    fg_reduce_group_kernel(const __grid_constant__ GroupParams P) {
  reduce_body<InterpProg<D, S>>(P);
}

template <class K>
static cudaError_t launch_one(K kernel, const GroupParams& p, int grid, int smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = pdl_config(grid, kThreads, smem, st);
  cudaLaunchAttribute at[1];
  pdl_attr(cfg, at);
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_group_kernel(const GroupParams& p, int exec, int big, int grid, int smem, cudaStream_t st) {
  if (exec == 0) {
    return big ? launch_one(fg_ew_group_kernel<8, 8>, p, grid, smem, st)
               : launch_one(fg_ew_group_kernel<4, 4>, p, grid, smem, st);
  }
  return big ? launch_one(fg_reduce_group_kernel<8, 8>, p, grid, smem, st)
             : launch_one(fg_reduce_group_kernel<4, 4>, p, grid, smem, st);
}

int group_kernel_threads() { return kThreads; }

}  // namespace fg
