// Host-callable kernel launchers (defined in the .cu files).
#pragma once
#include <cuda_runtime.h>

#include "fg_abi.h"

namespace fg {

// Launch configuration that lets a kernel be placed while the previous grid
// on the stream drains (programmatic dependent launch); every kernel here
// waits for that grid before its first global memory access.
inline cudaLaunchConfig_t pdl_config(int grid, int block, int smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  return cfg;
}
inline void pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&at)[1]) {
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
}

// exec: 0 = elementwise group (K1), 1 = reduce group (K2).  big selects the
// 8-register / 8-slot machine (one CTA per SM) over the 4/4 one.
cudaError_t launch_group_kernel(const GroupParams& p, int exec, int big, int grid, int smem, cudaStream_t st);
int group_kernel_threads();
// Records the message fg_last_error() returns on this thread; returns status.
int set_last_error(int status, const char* msg);

cudaError_t launch_gemm_kernel(const GemmParams& p, int big, int grid, int smem, cudaStream_t st);
// CTA pairs (2-CTA clusters) of the GEMM kernel's shape (one CTA per SM, `smem`
// bytes of shared memory) that the device runs at once; 0 if unknown.
int gemm_max_clusters(int smem);
int gemm_smem_bytes(const GemmParams& p);

// Tensor fusion.  One chunk = up to kTfChunk consecutive elements of one
// tensor; the tensor's last chunk also zeroes the padding after it.
constexpr int kTfChunk = 8192;
struct TfChunk {
  float* tensor;        // fp32 tensor base
  int64_t start;        // first element of the chunk
  int64_t buf_off;      // byte offset of element `start` in the fusion buffer
  int32_t count;        // elements in the chunk
  int32_t pad_bytes;    // bytes to zero after the chunk (last chunk of a tensor)
};
// Per-bucket readiness for a one-launch pack of several AllReduce buckets
// (all null otherwise): every chunk adds one to its bucket's count with a
// release reduction; the count is never reset.
struct TfBuckets {
  const int32_t* chunk_bucket = nullptr;   // bucket of every chunk of the launch
  const int32_t* nchunks = nullptr;        // chunks per bucket
  uint32_t* count = nullptr;               // chunks of the bucket written by every bucketed launch so far
                                           // (never reset; wraps modulo 2^32)
  uint32_t seq = 0;                        // this launch's number: bucket b is complete once count[b]
                                           // reaches seq * nchunks[b] (cyclic comparison)
  // observed launch: CTA 0 does not pack but watches the counts, in bucket
  // order, and writes to observe[b] the global timer when it saw bucket b
  // complete for launch seq + seq_offset (0 if it gave up after limit_ns,
  // with DEVERR_TIMEOUT in err); the packing CTAs write their latest
  // finishing time to observe[nb]
  unsigned long long* observe = nullptr;
  int32_t nb = 0;
  uint32_t seq_offset = 0;
  int64_t limit_ns = 0;
  int32_t* err = nullptr;
};
// claim: null = CTAs stride over the chunks; else the launch covers all of
// the layout's chunks and CTAs claim them from this counter (see the kernel)
// The pack CTAs that fit on nsm SMs at once (the grid of a claimed launch).
int tf_pack_resident(int nsm);
cudaError_t launch_tf_pack(const TfChunk* chunks, int nchunks, int buf_bf16, float scale, void* buf, int grid,
                           cudaStream_t st, const TfBuckets& bk = TfBuckets(), unsigned long long* claim = nullptr);
// Unpack runs one CTA per SM (grid = SM count); err receives DEVERR_TIMEOUT
// if a wait for a chunk load expires.
cudaError_t launch_tf_unpack(const TfChunk* chunks, int nchunks, int buf_bf16, float uscale, const void* buf,
                             int grid, int32_t* err, cudaStream_t st);

}  // namespace fg
