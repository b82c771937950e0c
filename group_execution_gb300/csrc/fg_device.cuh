// Device helpers for sm_103a: mbarriers with bounded waits, TMA tile copies,
// bulk-group bookkeeping, and the register-stack interpreter that runs a
// group's operator program on eight values per thread.
#pragma once
#ifndef __CUDACC_RTC__
#include <cstdint>
#include <cuda.h>
#endif

#include "fg_abi.h"

namespace fg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete, at most limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if ((int64_t)(global_ns() - t0) > limit_ns) return false;
  }
  return true;
}

// ---- TMA -------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const CUtensorMap* m, int32_t x, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2}], [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, int32_t x, int32_t y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(src)
               : "memory");
}
// Programmatic dependent launch: a grid lets the next grid on the stream be
// placed on the SMs while it drains, and waits, before its own first global
// memory access, for the previous grid to complete with its writes visible.
// Both are no-ops for a launch that did not ask for the overlap.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Contiguous copy global -> shared (both 16-byte aligned, bytes a multiple
// of 16), counted on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier over nthreads threads that also returns, to every one of
// them, whether any participant passed pred = true (one consistent decision).
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %3, 0;\n bar.red.or.pred q, %1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void set_error(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---- operator semantics (float32, one rounding per operator) -------------------
// Products and sums use the _rn intrinsics so the compiler never contracts
// two operators into one fused multiply-add: fusion must not change the
// per-operator rounding of the unfused program.
__device__ __forceinline__ float op_relu(float x) { return x > 0.f ? x : 0.f; }
__device__ __forceinline__ float op_sigmoid(float x) { return __frcp_rn(__fadd_rn(1.f, expf(-x))); }

// ---- the register-stack machine -------------------------------------------------
// V values per thread.  The top of the stack lives in TOP; the entries below
// it in R[0..D-2]; S save slots hold values a group reuses.  Unary operators
// and the leaf-operand forms act on TOP whatever the depth, so their code
// exists once; only moves between TOP, R and the slots depend on the depth,
// and those use compile-time register indices.  `Env` provides
// load_leaf(arg, float(&)[V]) and load_acc(float(&)[V]).
template <int D, int S, int V>
struct Machine {
  float TOP[V];
  float R[D > 1 ? D - 1 : 1][V];
  float SL[S > 0 ? S : 1][V];

  // push: the old top (stack depth d before the push, d >= 1) moves to R[d-1]
  template <int d>
  __device__ __forceinline__ void push(const float (&t)[V]) {
    if constexpr (d < D) {
      if constexpr (d >= 1) {
#pragma unroll
        for (int i = 0; i < V; ++i) R[d - 1][i] = TOP[i];
      }
#pragma unroll
      for (int i = 0; i < V; ++i) TOP[i] = t[i];
    }
  }
  // binary op at depth d: TOP = R[d-2] op TOP
  template <int op, int d>
  __device__ __forceinline__ void bin() {
    if constexpr (d >= 2 && d <= D) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const float a = R[d - 2][i], b = TOP[i];
        if constexpr (op == VM_ADD) TOP[i] = __fadd_rn(a, b);
        else if constexpr (op == VM_SUB) TOP[i] = __fsub_rn(a, b);
        else TOP[i] = __fmul_rn(a, b);
      }
    }
  }
  template <int d>
  __device__ __forceinline__ void second(float (&t)[V]) {
    if constexpr (d >= 2 && d <= D) {
#pragma unroll
      for (int i = 0; i < V; ++i) t[i] = R[d - 2][i];
    }
  }
  // The empty asm statements keep the compiler from merging the per-slot
  // cases into one indexed access, which would move the slots to local
  // memory.
  template <int op, int s>
  __device__ __forceinline__ void slot_bin(float (&t)[V]) {
    if constexpr (s < S) {
      asm volatile("");
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const float b = SL[s][i];
        if constexpr (op == VM_ADD_S) TOP[i] = __fadd_rn(TOP[i], b);
        else if constexpr (op == VM_SUB_S) TOP[i] = __fsub_rn(TOP[i], b);
        else if constexpr (op == VM_MUL_S) TOP[i] = __fmul_rn(TOP[i], b);
        else t[i] = b;
      }
    }
  }
  template <int s, int d>
  __device__ __forceinline__ void push_slot() {
    if constexpr (s < S && d < D) {
      asm volatile("");
      if constexpr (d >= 1) {
#pragma unroll
        for (int i = 0; i < V; ++i) R[d - 1][i] = TOP[i];
      }
#pragma unroll
      for (int i = 0; i < V; ++i) TOP[i] = SL[s][i];
    }
  }
  template <int s>
  __device__ __forceinline__ void tee() {
    if constexpr (s < S) {
      asm volatile("");
#pragma unroll
      for (int i = 0; i < V; ++i) SL[s][i] = TOP[i];
    }
  }
  // store: copy the top into slot s and pop (the entry below becomes TOP)
  template <int s, int d>
  __device__ __forceinline__ void store() {
    if constexpr (s < S && d >= 1 && d <= D) {
      asm volatile("");
#pragma unroll
      for (int i = 0; i < V; ++i) SL[s][i] = TOP[i];
      if constexpr (d >= 2) {
#pragma unroll
        for (int i = 0; i < V; ++i) TOP[i] = R[d - 2][i];
      }
    }
  }

  // Runs `n` instructions; the result is TOP.
  template <class Env>
  __device__ __forceinline__ void run(const VmInstr* prog, int n, Env& env) {
#pragma unroll 1
    for (int pc = 0; pc < n; ++pc) {
      const VmInstr ins = prog[pc];
      const int key = ins.key;
      float t[V];
      if (key < kCaseAcc || (key >= kCaseBinL && key < kCaseBinS)) env.load_leaf(ins.arg, t);
      else if (key < kCaseBin) env.load_acc(t);
      int dv = 0;   // 1: TOP = t / TOP, 2: TOP = TOP / t
      switch (key) {
#define FG_PUSH(d) \
  case kCaseLeaf + d: push<d>(t); break; \
  case kCaseAcc + d: push<d>(t); break;
#define FG_BIN(d) \
  case vm_case(VM_ADD, d, 0): bin<VM_ADD, d>(); break; \
  case vm_case(VM_SUB, d, 0): bin<VM_SUB, d>(); break; \
  case vm_case(VM_MUL, d, 0): bin<VM_MUL, d>(); break; \
  case vm_case(VM_DIV, d, 0): second<d>(t); dv = 1; break;
#define FG_SLOT_D(s, d) case vm_case(VM_PUSH_SLOT, d, s): push_slot<s, d>(); break;
#define FG_STORE_D(s, d) case vm_case(VM_STORE, d, s): store<s, d>(); break;
#define FG_SLOT(s) \
  case vm_case(VM_ADD_S, 0, s): slot_bin<VM_ADD_S, s>(t); break; \
  case vm_case(VM_SUB_S, 0, s): slot_bin<VM_SUB_S, s>(t); break; \
  case vm_case(VM_MUL_S, 0, s): slot_bin<VM_MUL_S, s>(t); break; \
  case vm_case(VM_DIV_S, 0, s): slot_bin<VM_DIV_S, s>(t); dv = 2; break; \
  case vm_case(VM_TEE, 0, s): tee<s>(); break; \
  FG_SLOT_D(s, 0) FG_SLOT_D(s, 1) FG_SLOT_D(s, 2) FG_SLOT_D(s, 3) \
  FG_SLOT_D(s, 4) FG_SLOT_D(s, 5) FG_SLOT_D(s, 6) FG_SLOT_D(s, 7) \
  FG_STORE_D(s, 1) FG_STORE_D(s, 2) FG_STORE_D(s, 3) FG_STORE_D(s, 4) \
  FG_STORE_D(s, 5) FG_STORE_D(s, 6) FG_STORE_D(s, 7) FG_STORE_D(s, 8)
        FG_PUSH(0) FG_PUSH(1) FG_PUSH(2) FG_PUSH(3) FG_PUSH(4) FG_PUSH(5) FG_PUSH(6) FG_PUSH(7)
        FG_BIN(2) FG_BIN(3) FG_BIN(4) FG_BIN(5) FG_BIN(6) FG_BIN(7) FG_BIN(8)
        case kCaseUn + (VM_SCALE - VM_SCALE):
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = __fmul_rn(ins.imm, TOP[i]);
          break;
        case kCaseUn + (VM_ADDC - VM_SCALE):
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = __fadd_rn(TOP[i], ins.imm);
          break;
        case kCaseUn + (VM_RELU - VM_SCALE):
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = op_relu(TOP[i]);
          break;
        case kCaseUn + (VM_EXP - VM_SCALE):
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = expf(TOP[i]);
          break;
        case kCaseUn + (VM_SIGMOID - VM_SCALE):
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = op_sigmoid(TOP[i]);
          break;
        case kCaseUn + (VM_TANH - VM_SCALE):
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = tanhf(TOP[i]);
          break;
        case kCaseUn + (VM_NEG - VM_SCALE):
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = -TOP[i];
          break;
        case kCaseBinL + 0:
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = __fadd_rn(TOP[i], t[i]);
          break;
        case kCaseBinL + 1:
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = __fsub_rn(TOP[i], t[i]);
          break;
        case kCaseBinL + 2:
#pragma unroll
          for (int i = 0; i < V; ++i) TOP[i] = __fmul_rn(TOP[i], t[i]);
          break;
        case kCaseBinL + 3: dv = 2; break;
        FG_SLOT(0) FG_SLOT(1) FG_SLOT(2) FG_SLOT(3) FG_SLOT(4) FG_SLOT(5) FG_SLOT(6) FG_SLOT(7)
#undef FG_SLOT
#undef FG_STORE_D
#undef FG_SLOT_D
#undef FG_BIN
#undef FG_PUSH
        default: break;
      }
      if (dv) {
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const float a = dv == 1 ? t[i] : TOP[i], b = dv == 1 ? TOP[i] : t[i];
          TOP[i] = __fdiv_rn(a, b);
        }
      }
    }
  }
};

}  // namespace fg

// ---- tcgen05 / TMEM ----------------------------------------------------------------
namespace fg {

// Allocates ncols TMEM columns (power of two >= 32); the address is written
// to shared memory at `dst`.  Executed by one whole warp; with CG = 2 by one
// warp in each CTA of the pair, which receive the same columns.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  if constexpr (CG == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma: start address, leading
// and stride byte offsets (all >> 4), the fixed 0b001 at bits 46-48, and the
// 128-byte swizzle mode (2) in bits 61-63.  Operand tiles are 1024-byte
// aligned, so the base-offset field stays 0.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A and B and an f32
// accumulator: D format bits 4-5 = 1 (f32), A format bits 7-9 = 1 (bf16),
// B format bits 10-12 = 1 (bf16), bit 15 / 16 = A / B major-ness (1 = MN),
// bits 17-22 = N >> 3, bits 24-28 = M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.  With CG = 2 the
// thread belongs to the even CTA of a pair and the instruction spans both
// SMs: each CTA supplies half of A's rows and half of B's columns at the same
// shared-memory offsets, and receives its half of D's rows in its own TMEM.
template <int CG>
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  if constexpr (CG == 1)
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on the mbarrier at `bar` in every CTA of the cluster whose bit
// is set in `mask` when every 2-SM MMA issued so far by this thread has
// completed (the pair's two CTAs: both producers get the ring slot back, both
// epilogues the accumulator).
__device__ __forceinline__ void tc_commit_mask(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(mask)
      : "memory");
}
// 32 consecutive f32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace fg

// ---- clusters -----------------------------------------------------------------------
namespace fg {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.aligned;\n barrier.cluster.wait.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// Arrival on an mbarrier that may live in another CTA of the cluster, as a
// signal (release at CTA scope: the signalled hazards, such as TMEM reads
// finished before tcgen05.fence::before_thread_sync, need no wider memory
// ordering, and a cluster-scope release also waits for this thread's bulk
// stores still in flight, about a microsecond).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Flags between CTAs: a release store after the data it publishes, an
// acquire load before the data it guards is read.
__device__ __forceinline__ void st_release_gpu(int32_t* p, int32_t v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// floor(x / d) for x < 2^31 by d's multiplier (FastDiv).
__device__ __forceinline__ uint32_t div_inv(uint32_t x, FastDiv f) {
  return (uint32_t)(((uint64_t)x * f.mul) >> f.sh);
}
// A gather's source offset, sum_k ((g / d_k) % m_k) * s_k, for g < 2^31.
template <class Desc>
__device__ __forceinline__ uint32_t digit_offset(const Desc& G, uint32_t g) {
  uint32_t f = 0;
  for (int q = 0; q < G.nterms; ++q) {
    const uint32_t a = div_inv(g, G.dd[q]);
    f += (a - div_inv(a, G.dm[q]) * (uint32_t)G.m[q]) * (uint32_t)G.s[q];
  }
  return f;
}

// A reduction with release semantics at GPU scope and no result: the thread
// does not wait for it.
__device__ __forceinline__ void red_add_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Counter increment that publishes the caller's earlier writes (release)
// and, to the thread that reads the last count, everyone's (acquire).
__device__ __forceinline__ int32_t atom_add_acq_rel_gpu(int32_t* p, int32_t v) {
  int32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Counter increment that only publishes the caller's earlier writes: later
// operations of the thread do not wait for it (its old value arrives in a
// register whenever the thread reads it).
__device__ __forceinline__ int32_t atom_add_release_gpu(int32_t* p, int32_t v) {
  int32_t old;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// L2 eviction policies for TMA copies: operand tiles that other tiles will
// read again stay (evict_last); data streamed once goes first (evict_first).
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (`cbar` is a cluster address), with
// an L2 eviction policy.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y,
                                                 uint32_t cbar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(cbar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y, int32_t z,
                                                 uint32_t cbar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(cbar), "l"(policy)
      : "memory");
}
// Hinted single-CTA loads and stores (GEMM epilogue streams).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* m, int32_t x, int32_t y, uint32_t src,
                                                  uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;"
               ::"l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(src), "l"(policy)
               : "memory");
}

}  // namespace fg
