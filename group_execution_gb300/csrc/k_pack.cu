// Tensor-fusion pack / unpack (K4 / K5): many small float32 gradient tensors
// to and from one contiguous fusion buffer in a single launch each (DisCo,
// Introduction, on tensor fusion: small tensors are combined into one whose
// size is the sum of theirs).
//
// The host splits every tensor into chunks of up to 4096 elements and uploads
// the chunk table once; CTAs stride over chunks.  Each thread moves 16
// elements per chunk: four 16-byte loads issued back to back, then the scaled,
// rounded values as 8- or 16-byte stores.  A tensor's last chunk also zeroes
// the padding up to the next aligned offset, so the buffer is fully defined.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"

namespace fg {

namespace {

constexpr int kPackThreads = 256;
constexpr int kPerThread = kTfChunk / kPackThreads;   // 16
static_assert(kPerThread == 16, "chunk geometry");

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void zero_pad(uint8_t* p, int bytes) {
  // padding never exceeds the alignment (<= a few hundred bytes); it starts
  // 2-byte aligned (bf16) or 4-byte aligned (f32)
  for (int i = threadIdx.x * 2; i < bytes; i += kPackThreads * 2) *reinterpret_cast<uint16_t*>(p + i) = 0;
}

__global__ void __launch_bounds__(kPackThreads) tf_pack_kernel(const TfChunk* __restrict__ chunks, int nchunks,
                                                               int bf16, float scale, uint8_t* __restrict__ buf) {
  for (int ci = blockIdx.x; ci < nchunks; ci += gridDim.x) {
    const TfChunk c = chunks[ci];
    const float* src = c.tensor + c.start;
    uint8_t* dst = buf + c.buf_off;
    const int e0 = threadIdx.x * 4;   // element offset of this thread's first float4
    if (c.count == kTfChunk) {
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = __ldcs(reinterpret_cast<const float4*>(src + e0 + k * 1024));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = __fmul_rn(v[k].x, scale), b = __fmul_rn(v[k].y, scale);
        const float cc = __fmul_rn(v[k].z, scale), d = __fmul_rn(v[k].w, scale);
        if (bf16) {
          *reinterpret_cast<uint2*>(dst + (size_t)(e0 + k * 1024) * 2) = make_uint2(pack2(a, b), pack2(cc, d));
        } else {
          *reinterpret_cast<float4*>(dst + (size_t)(e0 + k * 1024) * 4) = make_float4(a, b, cc, d);
        }
      }
    } else {
      for (int e = threadIdx.x; e < c.count; e += kPackThreads) {
        const float a = __fmul_rn(src[e], scale);
        if (bf16) {
          *reinterpret_cast<__nv_bfloat16*>(dst + (size_t)e * 2) = __float2bfloat16_rn(a);
        } else {
          *reinterpret_cast<float*>(dst + (size_t)e * 4) = a;
        }
      }
    }
    if (c.pad_bytes) zero_pad(dst + (size_t)c.count * (bf16 ? 2 : 4), c.pad_bytes);
  }
}

__global__ void __launch_bounds__(kPackThreads) tf_unpack_kernel(const TfChunk* __restrict__ chunks, int nchunks,
                                                                 int bf16, float uscale,
                                                                 const uint8_t* __restrict__ buf) {
  for (int ci = blockIdx.x; ci < nchunks; ci += gridDim.x) {
    const TfChunk c = chunks[ci];
    float* dst = c.tensor + c.start;
    const uint8_t* src = buf + c.buf_off;
    const int e0 = threadIdx.x * 4;
    if (c.count == kTfChunk) {
      if (bf16) {
        uint2 h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) h[k] = __ldcs(reinterpret_cast<const uint2*>(src + (size_t)(e0 + k * 1024) * 2));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = __uint_as_float(h[k].x << 16), b = __uint_as_float(h[k].x & 0xffff0000u);
          const float cc = __uint_as_float(h[k].y << 16), d = __uint_as_float(h[k].y & 0xffff0000u);
          __stcs(reinterpret_cast<float4*>(dst + e0 + k * 1024),
                 make_float4(__fmul_rn(a, uscale), __fmul_rn(b, uscale), __fmul_rn(cc, uscale), __fmul_rn(d, uscale)));
        }
      } else {
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldcs(reinterpret_cast<const float4*>(src + (size_t)(e0 + k * 1024) * 4));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          __stcs(reinterpret_cast<float4*>(dst + e0 + k * 1024),
                 make_float4(__fmul_rn(v[k].x, uscale), __fmul_rn(v[k].y, uscale), __fmul_rn(v[k].z, uscale),
                             __fmul_rn(v[k].w, uscale)));
      }
    } else {
      for (int e = threadIdx.x; e < c.count; e += kPackThreads) {
        float a;
        if (bf16) {
          const uint16_t h = *reinterpret_cast<const uint16_t*>(src + (size_t)e * 2);
          a = __uint_as_float((uint32_t)h << 16);
        } else {
          a = *reinterpret_cast<const float*>(src + (size_t)e * 4);
        }
        dst[e] = __fmul_rn(a, uscale);
      }
    }
  }
}

}  // namespace

cudaError_t launch_tf_pack(const TfChunk* chunks, int nchunks, int buf_bf16, float scale, void* buf, int grid,
                           cudaStream_t st) {
  tf_pack_kernel<<<grid, kPackThreads, 0, st>>>(chunks, nchunks, buf_bf16, scale, static_cast<uint8_t*>(buf));
  return cudaGetLastError();
}

cudaError_t launch_tf_unpack(const TfChunk* chunks, int nchunks, int buf_bf16, float uscale, const void* buf,
                             int grid, cudaStream_t st) {
  tf_unpack_kernel<<<grid, kPackThreads, 0, st>>>(chunks, nchunks, buf_bf16, uscale,
                                                  static_cast<const uint8_t*>(buf));
  return cudaGetLastError();
}

}  // namespace fg
