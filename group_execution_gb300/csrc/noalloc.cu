// Row reduction that allocates no device memory.
//
// Some callers cannot call cudaMalloc at the point where they need a
// reduction: a host framework that owns every device allocation through its
// own pool and forbids direct allocations, or a latency-critical step where
// the device-wide synchronisation an allocation may imply is not acceptable.
// They also cannot build a plan (a plan owns device tables).  This entry
// point runs the reduce-group kernel on a one-operator program with its
// scratch (per-split partial row values and per-strip arrival counters) in a
// file-scope device array instead of plan-owned memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "groupexec.h"
#include "launch.h"

namespace fg {
namespace {

// Limits of the shared scratch: at most 65536 rows and 16 column splits.
constexpr int64_t kMaxRows = 65536;
constexpr int kMaxSplits = 16;
constexpr size_t kPartialBytes = size_t(kMaxRows) * kMaxSplits * sizeof(float);   // 4 MiB
constexpr size_t kCounterBytes = size_t(kMaxRows / kTileR) * sizeof(int32_t);     // 8 KiB
constexpr size_t kErrOffset = kPartialBytes + kCounterBytes;                          // the error word
constexpr size_t kScratchBytes = kErrOffset + 256;

// Held by every GPU that loads the library until the process exits.  All
// calls share it: calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on it.  Layout: partial row
// values | arrival counters | one error word that a kernel giving up on a
// bounded wait latches, read and cleared by fg_row_reduce_noalloc_status.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
constexpr int kMaxDevices = 64;
// The array's device address per device, and the context it was looked up
// in: a context that is destroyed and created again (cudaDeviceReset) loads
// the module again, possibly at another address, so the lookup is redone
// when the current context's id changes.
struct ScratchAddr {
  unsigned long long ctx_id;
  void* addr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

template <class Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  return nullptr;
}

// Id of the calling thread's current context (0 if there is none yet or it
// cannot be read: the lookup below then runs, and makes the device's primary
// context current).
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_ctx = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_ctx || !get_id || get_ctx(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device.  The first call
// on a device (per host thread that has no current context yet), and the
// first after the device's context was created again, looks it up.
void* scratch_address(int dev, cudaError_t* e) {
  const unsigned long long id = current_ctx_id();
  std::lock_guard<std::mutex> g(g_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  if (!a.addr || id == 0 || a.ctx_id != id) {
    void* p = nullptr;
    *e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*e != cudaSuccess) return nullptr;
    a.addr = p;
    a.ctx_id = id;
  }
  *e = cudaSuccess;
  return a.addr;
}

}  // namespace
}  // namespace fg

using namespace fg;

extern "C" fg_status fg_row_reduce_noalloc(int32_t opcode, const float* x, int64_t rows, int64_t cols, float* y,
                                           void* cuda_stream) {
  if (opcode != FG_OP_ROWSUM && opcode != FG_OP_ROWMAX)
    return (fg_status)set_last_error(FG_EINVAL, "opcode must be FG_OP_ROWSUM or FG_OP_ROWMAX");
  if (!x || !y) return (fg_status)set_last_error(FG_EINVAL, "null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(y) % 4)
    return (fg_status)set_last_error(FG_EINVAL, "x must be 16-byte and y 4-byte aligned");
  if (rows < 1 || cols < 1) return (fg_status)set_last_error(FG_ESHAPE, "empty matrix");
  if (rows > kMaxRows)
    return (fg_status)set_last_error(FG_EINVAL, "rows exceed the 65536-row limit of the no-allocation scratch");
  if (cols >= (int64_t(1) << 31) || rows * cols >= (int64_t(1) << 31))
    return (fg_status)set_last_error(FG_ESHAPE, "matrix of 2^31 or more elements");
  int dev = 0, nsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess || dev >= kMaxDevices)
    return (fg_status)set_last_error(FG_ECUDA, "no usable CUDA device");
  uint8_t* scratch = static_cast<uint8_t*>(scratch_address(dev, &e));
  if (!scratch) return (fg_status)set_last_error(FG_ECUDA, cudaGetErrorString(e));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);

  GroupParams p;
  std::memset(&p, 0, sizeof(p));
  p.prog[0] = VmInstr{(uint16_t)vm_case(VM_PUSH_LEAF, 0, 0), 0, 0.f};
  p.nprog = 1;
  p.nleaves = 1;
  p.FR = (int32_t)rows;
  p.FC = (int32_t)cols;
  p.ntr = (int32_t)((rows + kTileR - 1) / kTileR);
  p.ntc = (int32_t)((cols + kTileC - 1) / kTileC);
  p.ntiles = p.ntr * p.ntc;
  p.out = y;
  p.red_op = opcode == FG_OP_ROWSUM ? RED_SUM : RED_MAX;
  p.wait_limit_ns = 2000000000LL;
  LeafDesc& L = p.leaves[0];
  L.ptr = x;
  L.map_idx = 0;
  L.stage_off = 0;
  if (cols % 4 == 0) {
    // the row is staged through shared memory by TMA
    L.cls = LEAF_IDENT;
    EncodeFn enc = encoder();
    if (!enc) return (fg_status)set_last_error(FG_ECUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows}, strides[1] = {(cuuint64_t)cols * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)kTileR}, es[2] = {1, 1};
    if (enc(&p.maps[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return (fg_status)set_last_error(FG_ECUDA, "cuTensorMapEncodeTiled failed");
    p.stage_bytes = p.tx_bytes = kTileR * kTileC * 4;
    p.nstages = 12;
  } else {
    // rows not 16-byte aligned: each element is loaded directly
    L.cls = LEAF_GATHER;
    L.nterms = 1;
    L.d[0] = 1;
    L.m[0] = rows * cols;
    L.s[0] = 1;
    L.dd[0] = fast_div(1);
    L.dm[0] = fast_div(rows * cols);
    p.stage_bytes = p.tx_bytes = 0;
    p.nstages = 4;
  }
  // column splits: enough work units for every SM, at most 16 splits
  const int want = 4 * nsm;
  int nsplit = (want + p.ntr - 1) / p.ntr;
  nsplit = nsplit < 1 ? 1 : nsplit;
  nsplit = nsplit > kMaxSplits ? kMaxSplits : nsplit;
  const int cap = p.ntc / 16 > 1 ? p.ntc / 16 : 1;
  nsplit = nsplit > cap ? cap : nsplit;
  const int tps = (p.ntc + nsplit - 1) / nsplit;
  nsplit = (p.ntc + tps - 1) / tps;
  p.nsplit = nsplit;
  p.tiles_per_split = tps;
  p.nunits = p.ntr * nsplit;
  p.scratch = reinterpret_cast<float*>(scratch);
  p.counters = reinterpret_cast<int32_t*>(scratch + kPartialBytes);
  p.err = reinterpret_cast<int32_t*>(scratch + kErrOffset);
  // the arrival counters must start at zero (a call cut short by a device
  // timeout could leave them set); partial values are written before read
  if (nsplit > 1) {
    e = cudaMemsetAsync(p.counters, 0, sizeof(int32_t) * (size_t)p.ntr, st);
    if (e != cudaSuccess) return (fg_status)set_last_error(FG_ECUDA, cudaGetErrorString(e));
  }
  const int smem = 2048 + 2 * kConsumerWarps * 32 * 4 + p.nstages * p.stage_bytes;
  int grid = 2 * nsm;
  if (grid > p.nunits) grid = p.nunits;
  e = launch_group_kernel(p, 1, 0, grid, smem, st);
  if (e != cudaSuccess) return (fg_status)set_last_error(FG_ECUDA, cudaGetErrorString(e));
  return FG_OK;
}

extern "C" fg_status fg_row_reduce_noalloc_status(void* cuda_stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev >= kMaxDevices)
    return (fg_status)set_last_error(FG_ECUDA, "no usable CUDA device");
  uint8_t* scratch = static_cast<uint8_t*>(scratch_address(dev, &e));
  if (!scratch) return (fg_status)set_last_error(FG_ECUDA, cudaGetErrorString(e));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return (fg_status)set_last_error(FG_ECUDA, cudaGetErrorString(e));
  int32_t word = 0;
  e = cudaMemcpyAsync(&word, scratch + kErrOffset, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return (fg_status)set_last_error(FG_ECUDA, cudaGetErrorString(e));
  if (word == 0) return FG_OK;
  e = cudaMemsetAsync(scratch + kErrOffset, 0, sizeof(word), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return (fg_status)set_last_error(FG_ECUDA, cudaGetErrorString(e));
  if (word == DEVERR_TIMEOUT)
    return (fg_status)set_last_error(FG_ETIMEOUT, "a device-side wait of fg_row_reduce_noalloc exceeded 2 s");
  return (fg_status)set_last_error(FG_EDEVICE, ("device error word " + std::to_string(word)).c_str());
}
