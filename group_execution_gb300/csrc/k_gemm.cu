// The interpreted variants of the GEMM-epilogue kernel (the compiled
// variants share gemm_kernel.cuh through jit.cpp).
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"
#include "launch.h"

namespace fg {

template <int D, int S>
__global__ void __cluster_dims__(kGemmCluster, 1, 1) __launch_bounds__(kGemmThreads, 1)
    fg_gemm_epi_kernel(const __grid_constant__ GemmParams P) {
  gemm_body<InterpGemmEpi<D, S>, kGemmCluster>(P);
}

cudaError_t launch_gemm_kernel(const GemmParams& p, int big, int grid, int smem, cudaStream_t st) {
  auto k = big ? fg_gemm_epi_kernel<8, 8> : fg_gemm_epi_kernel<4, 4>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kGemmThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace fg
