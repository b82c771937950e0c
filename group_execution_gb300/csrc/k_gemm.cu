// The interpreted variants of the GEMM-epilogue kernel (the compiled
// variants share gemm_kernel.cuh through jit.cpp).
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"
#include "launch.h"

namespace fg {

template <int D, int S>
__global__ void __cluster_dims__(kGemmCluster, 1, 1) __launch_bounds__(kGemmThreads, 1)
    fg_gemm_epi_kernel(const __grid_constant__ GemmParams P) {
  gemm_body<InterpGemmEpi<D, S>, kGemmKB, kGemmN>(P);
}

cudaError_t launch_gemm_kernel(const GemmParams& p, int big, int grid, int smem, cudaStream_t st) {
  auto k = big ? fg_gemm_epi_kernel<8, 8> : fg_gemm_epi_kernel<4, 4>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = pdl_config(grid, kGemmThreads, smem, st);
  cudaLaunchAttribute at[1];
  pdl_attr(cfg, at);
  return cudaLaunchKernelEx(&cfg, k, p);
}

// Stands in for the GEMM kernel in the occupancy query: residency is set by
// the shared memory (more than half an SM's) and the pair clusters.
__global__ void __launch_bounds__(kGemmThreads, 1) fg_gemm_residency_probe(int) {}

int gemm_max_clusters(int smem) {
  static int cached[256] = {};   // [smem / 1 KB]: pairs + 1
  const int si = (smem >> 10) & 255;
  if (cached[si]) return cached[si] - 1;
  if (cudaFuncSetAttribute(fg_gemm_residency_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kGemmCluster);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kGemmCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fg_gemm_residency_probe, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached[si] = n + 1;
  return n;
}

}  // namespace fg
