// Tensor-fusion pack / unpack (K4 / K5): many small float32 gradient tensors
// to and from one contiguous fusion buffer in a single launch each (DisCo,
// Introduction, on tensor fusion: small tensors are combined into one whose
// size is the sum of theirs).
//
// The host splits every tensor into chunks of up to 8192 elements and uploads
// the chunk table once.  Pack: each CTA starts on a fixed chunk and then
// either strides over the chunks (range packs) or claims the next one from a
// layout counter (packs of the whole layout, bucketed or not); each thread
// issues all of its loads for a full chunk (32 elements, 128 bytes) before
// any conversion, and the next chunk's descriptor is fetched while the
// current chunk is in flight.  A tensor's last chunk also zeroes the padding
// up to the next aligned offset, so the buffer is fully defined.  Unpack: one
// CTA per SM; a producer warp brings chunks of the buffer into a
// shared-memory ring with bulk copies (rounded up to 16 bytes, which stays
// inside the tensor's padding), four warps widen and scale them into a
// staging buffer, and each chunk leaves as one bulk store of its 16-byte
// multiple plus at most three plain stores.
//
// A pack of several AllReduce buckets in one launch counts every chunk it
// writes into its bucket's count with a release reduction.  The counts are
// never reset: the k-th launch has completed bucket b once b's count reaches
// k times b's chunk count, so a stream-ordered wait can start that bucket's
// AllReduce while the rest is still being packed.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cuda_runtime.h>

#include "fg_device.cuh"
#include "launch.h"

namespace fg {

namespace {

constexpr int kPackThreads = 256;     // pack: 32 elements (128 bytes of loads) per thread
static_assert(kTfChunk == 32 * kPackThreads, "chunk geometry");

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void zero_pad(uint8_t* p, int bytes) {
  // padding never exceeds the alignment; it starts 2-byte aligned (bf16) or
  // 4-byte aligned (f32)
  for (int i = threadIdx.x * 2; i < bytes; i += kPackThreads * 2) *reinterpret_cast<uint16_t*>(p + i) = 0;
}

// The observer of an observed launch (one thread): each bucket's count, in
// bucket order, read with acquire until it reaches the watched launch's
// total, each wait bounded.
__device__ void observe_buckets(const TfBuckets& bk) {
  bool dead = false;
  for (int b = 0; b < bk.nb; ++b) {
    const uint32_t want = (bk.seq + bk.seq_offset) * (uint32_t)bk.nchunks[b];
    unsigned long long t = 0;
    if (!dead) {
      const uint64_t t0 = global_ns();
      for (;;) {
        const uint32_t v = (uint32_t)ld_acquire_gpu(reinterpret_cast<const int32_t*>(bk.count + b));
        const uint64_t now = global_ns();
        if ((int32_t)(v - want) >= 0) {
          t = now;
          break;
        }
        if ((int64_t)(now - t0) > bk.limit_ns) {
          dead = true;
          set_error(bk.err, DEVERR_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    bk.observe[b] = t;
  }
}

// claim: null = CTAs stride over the chunks; else each CTA's first chunk is
// fixed and the next ones are claimed from this counter, which a launch
// advances by exactly nchunks (each CTA with a first chunk claims until one
// claim fails), so that claim c is chunk ncta + c mod nchunks.  SMs do not
// stream at the same rate: claiming keeps every CTA busy until the chunks run
// out.
__global__ void __launch_bounds__(kPackThreads) tf_pack_kernel(const TfChunk* __restrict__ chunks, int nchunks,
                                                               int bf16, float scale, uint8_t* __restrict__ buf,
                                                               const TfBuckets bk, unsigned long long* claim) {
  __shared__ int s_nx[2];
  __shared__ TfChunk s_cn[2];
  pdl_launch_dependents();
  pdl_wait();   // the previous grid's writes are visible from here on
  // an observed launch: CTA 0 watches the buckets, the others pack
  const int obs = bk.observe ? 1 : 0;
  if (obs && blockIdx.x == 0) {
    if (threadIdx.x == 0) observe_buckets(bk);
    return;
  }
  const int cta = (int)blockIdx.x - obs, ncta = (int)gridDim.x - obs;
  int ci = cta;
  if (ci >= nchunks) return;
  TfChunk c = chunks[ci];
  for (int it = 0;; ++it) {
    int nx = ci + ncta;
    TfChunk cn;
    unsigned long long cl = 0;
    if (claim) {
      if (threadIdx.x == 0) cl = atomicAdd(claim, 1ull);   // the next chunk, in flight meanwhile
    } else if (nx < nchunks) {
      cn = chunks[nx];
    }
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
    if (claim) {
      // thread 0 shares the claimed chunk (buffers alternate, so a thread
      // still reading the last one is never overwritten)
      if (threadIdx.x == 0) {
        const int n2 = ncta + (int)(cl % (unsigned long long)nchunks);
        s_nx[it & 1] = n2;
        if (n2 < nchunks) s_cn[it & 1] = chunks[n2];
      }
      __syncthreads();
      nx = s_nx[it & 1];
      if (nx < nchunks) cn = s_cn[it & 1];
    }
    if (bk.count) {
      // count the chunk for its bucket: the barrier orders every thread's
      // stores before thread 0's release reduction (cumulative), which
      // returns nothing, so thread 0 does not wait for it; a reader that
      // sees the bucket's total with acquire sees every chunk counted
      if (!claim) __syncthreads();
      if (threadIdx.x == 0) red_add_release_gpu(bk.count + bk.chunk_bucket[ci], 1u);
    }
    if (nx >= nchunks) break;
    ci = nx;
    c = cn;
  }
  if (obs && threadIdx.x == 0) atomicMax(bk.observe + bk.nb, (unsigned long long)global_ns());
}

constexpr int kUnpackConsumers = 128;                  // four warps
constexpr int kUnpackThreadsTma = 32 + kUnpackConsumers;  // + the producer warp
constexpr int kUnpackOutBufs = 4;
constexpr int kUnpackOutBytes = kTfChunk * 4;
constexpr int64_t kUnpackWaitNs = 100000000LL;          // 100 ms: a chunk load never takes this long

// Stages of the load ring: bf16 chunks are 16 KB, f32 chunks 32 KB.
__host__ __device__ constexpr int unpack_stages(int bf16) { return bf16 ? 4 : 3; }

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(kUnpackThreadsTma, 1)
    tf_unpack_kernel(const TfChunk* __restrict__ chunks, int nchunks, int bf16, float uscale,
                     const uint8_t* __restrict__ buf, int32_t* err) {
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 127) & ~uintptr_t(127));
  const int NS = unpack_stages(bf16);
  const int stage_bytes = kTfChunk * (bf16 ? 2 : 4);
  const uint32_t full0 = smem_u32(sm), empty0 = full0 + 64;
  uint8_t* stage0 = sm + 128;
  uint8_t* out0 = stage0 + NS * stage_bytes;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();   // the previous grid's writes are visible from here on
  const int warp = threadIdx.x >> 5;

  if (warp == 0) {
    // ---- producer: one bulk copy per chunk ----
    if (threadIdx.x == 0) {
      int k = 0;
      bool ok = true;
      for (int ci = blockIdx.x; ci < nchunks; ci += gridDim.x, ++k) {
        const int s = k % NS;
        if (k >= NS && !mbar_wait(empty0 + 8 * s, ((k / NS) & 1) ^ 1, kUnpackWaitNs)) {
          ok = false;
          break;
        }
        const TfChunk c = chunks[ci];
        // a partial chunk's bytes rounded up to 16 end inside its padding
        const uint32_t bytes = ((uint32_t)c.count * (bf16 ? 2u : 4u) + 15u) & ~15u;
        if (bytes) {
          mbar_expect_tx(full0 + 8 * s, bytes);
          bulk_load(smem_u32(stage0 + s * stage_bytes), buf + c.buf_off, bytes, full0 + 8 * s);
        } else {
          mbar_arrive(full0 + 8 * s);   // an empty tensor
        }
      }
      if (!ok) {
        // the consumers' own bounded waits end their loop
        set_error(err, DEVERR_TIMEOUT);
        for (int j = k - NS < 0 ? 0 : k - NS; j < k; ++j) mbar_wait(full0 + 8 * (j % NS), (j / NS) & 1, kUnpackWaitNs);
      }
    }
  } else {
    // ---- consumers ----
    const int t = threadIdx.x - 32;
    int k = 0;
    bool failed = false;
    for (int ci = blockIdx.x; ci < nchunks; ci += gridDim.x, ++k) {
      const int s = k % NS;
      const TfChunk c = chunks[ci];
      const bool got = mbar_wait(full0 + 8 * s, (k / NS) & 1, kUnpackWaitNs);
      uint8_t* ob = out0 + (k % kUnpackOutBufs) * kUnpackOutBytes;
      if (got) {
        const uint8_t* st = stage0 + s * stage_bytes;
        const int ngroups = (c.count + 3) >> 2;   // groups of 4 elements (the last may be partial)
        // consecutive threads take consecutive groups (conflict-free
        // shared-memory accesses)
#pragma unroll 4
        for (int g = t; g < ngroups; g += kUnpackConsumers) {
          float4 f;
          if (bf16) {
            const uint2 h = *reinterpret_cast<const uint2*>(st + g * 8);
            f = make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xffff0000u),
                            __uint_as_float(h.y << 16), __uint_as_float(h.y & 0xffff0000u));
          } else {
            f = *reinterpret_cast<const float4*>(st + g * 16);
          }
          *reinterpret_cast<float4*>(ob + g * 16) =
              make_float4(__fmul_rn(f.x, uscale), __fmul_rn(f.y, uscale), __fmul_rn(f.z, uscale),
                          __fmul_rn(f.w, uscale));
        }
        fence_proxy_async_smem();
      }
      // the staging buffer the next chunk writes was last stored kUnpackOutBufs
      // chunks ago: at most kUnpackOutBufs - 2 newer stores may still read
      if (t == 0) bulk_wait_read<kUnpackOutBufs - 2>();
      // every consumer takes the same decision: stop if any wait expired
      failed = named_bar_or(1, kUnpackConsumers, !got);
      if (failed) break;
      if (t == 0) {
        float* dst = c.tensor + c.start;
        const int body = c.count & ~3;
        if (body > 0) bulk_store(dst, smem_u32(ob), (uint32_t)body * 4u);
        bulk_commit();
        for (int e = body; e < c.count; ++e) dst[e] = reinterpret_cast<const float*>(ob)[e];
        mbar_arrive(empty0 + 8 * s);
      }
    }
    if (failed && t == 0) set_error(err, DEVERR_TIMEOUT);
    if (t == 0) bulk_wait<0>();
  }
}

}  // namespace

cudaError_t launch_tf_pack(const TfChunk* chunks, int nchunks, int buf_bf16, float scale, void* buf, int grid,
                           cudaStream_t st, const TfBuckets& bk, unsigned long long* claim) {
  cudaLaunchConfig_t cfg = pdl_config(grid, kPackThreads, 0, st);
  cudaLaunchAttribute at[1];
  pdl_attr(cfg, at);
  return cudaLaunchKernelEx(&cfg, tf_pack_kernel, chunks, nchunks, buf_bf16, scale, static_cast<uint8_t*>(buf), bk,
                            claim);
}

int tf_pack_resident(int nsm) {
  // A claimed launch fixes each CTA's first chunk, so every CTA of its grid
  // must be resident from the start: one that waits for a slot would only
  // start once the others run out of chunks, with its first chunk last.
  static std::atomic<int> per_sm{0};
  int k = per_sm.load(std::memory_order_relaxed);
  if (!k) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, tf_pack_kernel, kPackThreads, 0) != cudaSuccess || k < 1) {
      (void)cudaGetLastError();
      return nsm;
    }
    per_sm.store(k, std::memory_order_relaxed);
  }
  return k * nsm;
}

int tf_unpack_smem(int buf_bf16) {
  return 128 + 128 + unpack_stages(buf_bf16) * kTfChunk * (buf_bf16 ? 2 : 4) + kUnpackOutBufs * kUnpackOutBytes;
}

cudaError_t launch_tf_unpack(const TfChunk* chunks, int nchunks, int buf_bf16, float uscale, const void* buf,
                             int grid, int32_t* err, cudaStream_t st) {
  const int smem = tf_unpack_smem(buf_bf16);
  // the shared-memory opt-in is set once per device (the largest size either
  // buffer type needs), not on every launch
  static std::atomic<uint64_t> opted{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(opted.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(tf_unpack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             std::max(tf_unpack_smem(0), tf_unpack_smem(1)));
    if (e != cudaSuccess) return e;
    opted.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = pdl_config(grid, kUnpackThreadsTma, smem, st);
  cudaLaunchAttribute at[1];
  pdl_attr(cfg, at);
  return cudaLaunchKernelEx(&cfg, tf_unpack_kernel, chunks, nchunks, buf_bf16, uscale, static_cast<const uint8_t*>(buf), err);
}

}  // namespace fg
