// Tensor-fusion pack / unpack (K4 / K5): many small float32 gradient tensors
// to and from one contiguous fusion buffer in a single launch each (DisCo,
// Introduction, on tensor fusion: small tensors are combined into one whose
// size is the sum of theirs).
//
// The host splits every tensor into chunks of up to 8192 elements and uploads
// the chunk table once; CTAs stride over chunks.  Each thread issues all of
// its loads for a full chunk (32 elements: 128 bytes when packing, 64 bytes
// when unpacking bf16) before any conversion, and the next chunk's
// descriptor is fetched while the current chunk is in flight.  A tensor's last chunk also zeroes the padding
// up to the next aligned offset, so the buffer is fully defined.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"

namespace fg {

namespace {

constexpr int kPackThreads = 256;     // pack: 32 elements (128 bytes of loads) per thread
constexpr int kUnpackThreads = 256;   // unpack: 32 bf16 elements (64 bytes of loads) per thread
static_assert(kTfChunk == 32 * kPackThreads && kTfChunk == 32 * kUnpackThreads, "chunk geometry");

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void zero_pad(uint8_t* p, int bytes) {
  // padding never exceeds the alignment; it starts 2-byte aligned (bf16) or
  // 4-byte aligned (f32)
  for (int i = threadIdx.x * 2; i < bytes; i += kPackThreads * 2) *reinterpret_cast<uint16_t*>(p + i) = 0;
}

__global__ void __launch_bounds__(kPackThreads) tf_pack_kernel(const TfChunk* __restrict__ chunks, int nchunks,
                                                               int bf16, float scale, uint8_t* __restrict__ buf) {
  int ci = blockIdx.x;
  if (ci >= nchunks) return;
  TfChunk c = chunks[ci];
  for (; ci < nchunks; ci += gridDim.x) {
    const int nx = ci + gridDim.x;
    TfChunk cn;
    if (nx < nchunks) cn = chunks[nx];
    const float* src = c.tensor + c.start;
    uint8_t* dst = buf + c.buf_off;
    if (c.count == kTfChunk) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __ldcs(reinterpret_cast<const float4*>(src) + threadIdx.x + k * kPackThreads);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int e = 4 * (threadIdx.x + k * kPackThreads);
        const float a = __fmul_rn(v[k].x, scale), b = __fmul_rn(v[k].y, scale);
        const float cc = __fmul_rn(v[k].z, scale), d = __fmul_rn(v[k].w, scale);
        if (bf16) {
          *reinterpret_cast<uint2*>(dst + (size_t)e * 2) = make_uint2(pack2(a, b), pack2(cc, d));
        } else {
          *reinterpret_cast<float4*>(dst + (size_t)e * 4) = make_float4(a, b, cc, d);
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
    c = cn;
  }
}

__global__ void __launch_bounds__(kUnpackThreads) tf_unpack_kernel(const TfChunk* __restrict__ chunks, int nchunks,
                                                                 int bf16, float uscale,
                                                                 const uint8_t* __restrict__ buf) {
  int ci = blockIdx.x;
  if (ci >= nchunks) return;
  TfChunk c = chunks[ci];
  for (; ci < nchunks; ci += gridDim.x) {
    const int nx = ci + gridDim.x;
    TfChunk cn;
    if (nx < nchunks) cn = chunks[nx];
    float* dst = c.tensor + c.start;
    const uint8_t* src = buf + c.buf_off;
    if (c.count == kTfChunk && bf16) {
      // 8 bf16 (16 bytes) per load, four loads per thread
      uint4 h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = __ldcs(reinterpret_cast<const uint4*>(src) + threadIdx.x + k * kUnpackThreads);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = 8 * (threadIdx.x + k * kUnpackThreads);
        const uint32_t w[4] = {h[k].x, h[k].y, h[k].z, h[k].w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f[2 * j] = __fmul_rn(__uint_as_float(w[j] << 16), uscale);
          f[2 * j + 1] = __fmul_rn(__uint_as_float(w[j] & 0xffff0000u), uscale);
        }
        __stcs(reinterpret_cast<float4*>(dst + e), make_float4(f[0], f[1], f[2], f[3]));
        __stcs(reinterpret_cast<float4*>(dst + e) + 1, make_float4(f[4], f[5], f[6], f[7]));
      }
    } else if (c.count == kTfChunk) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[k] = __ldcs(reinterpret_cast<const float4*>(src) + threadIdx.x + (half * 4 + k) * kUnpackThreads);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          __stcs(reinterpret_cast<float4*>(dst) + threadIdx.x + (half * 4 + k) * kUnpackThreads,
                 make_float4(__fmul_rn(v[k].x, uscale), __fmul_rn(v[k].y, uscale), __fmul_rn(v[k].z, uscale),
                             __fmul_rn(v[k].w, uscale)));
      }
    } else {
      for (int e = threadIdx.x; e < c.count; e += kUnpackThreads) {
        float a;
        if (bf16) {
          const uint16_t hh = *reinterpret_cast<const uint16_t*>(src + (size_t)e * 2);
          a = __uint_as_float((uint32_t)hh << 16);
        } else {
          a = *reinterpret_cast<const float*>(src + (size_t)e * 4);
        }
        dst[e] = __fmul_rn(a, uscale);
      }
    }
    c = cn;
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
  tf_unpack_kernel<<<grid, kUnpackThreads, 0, st>>>(chunks, nchunks, buf_bf16, uscale,
                                                  static_cast<const uint8_t*>(buf));
  return cudaGetLastError();
}

}  // namespace fg
