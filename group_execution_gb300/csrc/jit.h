// Plan-build-time compilation of group programs (see jit.cpp).
#pragma once
#include <cuda_runtime.h>

#include <functional>
#include <string>
#include <vector>

#include "host.h"

namespace fg {

bool jit_available();
// CUDA source of a group's kernel; min_blocks is the kernel's CTAs-per-SM bound.
// small_seg > 0: also the direct kernel (direct leaf reads), fg_jit_small_group,
// for that many warps per frame row (its segmented body when more than one)
std::string jit_source(const CompiledGroup& cg, int min_blocks, int small_seg = 0);
// Compiles (once per process per distinct source) and loads; returns "" or an
// error message.  funcs[i] is the loaded kernel of sources[i].
std::string jit_compile(const std::vector<std::string>& sources, std::vector<void*>& funcs,
                        std::vector<void*>* small_funcs = nullptr);
// One launch of a compiled kernel with `params` as its only argument; pdl:
// the launch may begin while the stream's previous kernel finishes (the
// kernel waits for it with griddepcontrol.wait).
cudaError_t jit_launch_any(void* func, void* params, int grid, int threads, int smem, cudaStream_t st,
                           bool pdl = true);
cudaError_t jit_launch(void* func, const GroupParams& p, int grid, int smem, cudaStream_t st);
cudaError_t jit_launch_gemm(void* func, const GemmParams& p, int grid, int smem, cudaStream_t st);

}  // namespace fg
