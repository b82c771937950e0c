// Fused-group kernels for elementwise/broadcast/injective groups (K1) and
// groups ending in a row reduction (K2), templated on how the group's
// operator program is evaluated: `Prog` is either the register-stack
// interpreter (InterpProg) or a straight-line program generated from the
// group and compiled at plan-build time.
//
// Persistent CTAs (one per SM slot) walk 32x64 tiles of the group's frame.
// Two producer warps, taking alternate ring stages, stream every staged
// leaf's tile into a ring of shared-memory stages with TMA (transposed leaves
// arrive as transposed boxes, so the transposition costs no extra global
// traffic); eight consumer warps evaluate the program on the tile from
// shared memory, eight values per thread, in registers.  K1 writes the
// result with TMA stores and claims its tiles from a per-group counter; K2
// folds it into per-row partial sums or maxima.  No intermediate of the
// group ever reaches global memory (TVM "Operator Fusion", FuseTIR; DisCo,
// Introduction, on op fusion).  Small groups and row reductions over
// row-contiguous leaves run the direct kernel at the end of this file
// instead.
//
// Thread layout inside a tile: lane = tile row (0..31), consumer warp w owns
// tile columns 8w..8w+7.  Staged 2-D boxes are 128-byte swizzled so that the
// row-per-lane reads (and the column-per-lane reads of transposed boxes) hit
// 32 distinct banks.
#pragma once
#include "fg_device.cuh"

namespace fg {

constexpr int kThreads = (kConsumerWarps + kProducerWarps) * 32;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kOutBufBytes = kTileR * kTileC * 4;   // 8 KB
constexpr int kXOutSliceBytes = kOutBufBytes;        // per extra output: 8 warps x 32 x 8 floats

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<uint8_t*>((a + 1023) & ~uintptr_t(1023));
}

// Bounded wait that also gives up as soon as another thread of the CTA has
// recorded a timeout.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, int64_t limit,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if ((int64_t)(global_ns() - t0) > limit) return false;
  }
  return true;
}

// 128-byte swizzled address of (row, 16-byte chunk) inside a box whose rows
// are 128 bytes long.
__device__ __forceinline__ int swz(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

// ---- leaf reads for one thread: 8 frame points (r0+lr, c0+lc0 .. c0+lc0+7) ----
struct TileEnv {
  const GroupParams& P;
  const uint8_t* stage;
  int lr, lc0, r0, c0;
  uint8_t* xb = nullptr;   // this warp's staging slices of the extra outputs (TMA stores), or none

  __device__ __forceinline__ void ident(int off, float (&t)[8]) const {
    const uint8_t* b = stage + off + (lc0 >> 5) * (kTileR * 128);
    const int j0 = (lc0 & 31) >> 2;
    const float4 a = *reinterpret_cast<const float4*>(b + swz(lr, j0));
    const float4 c = *reinterpret_cast<const float4*>(b + swz(lr, j0 + 1));
    t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w;
    t[4] = c.x; t[5] = c.y; t[6] = c.z; t[7] = c.w;
  }
  // box rows are frame columns, 32 frame rows per 128-byte box row
  __device__ __forceinline__ void trans(int off, float (&t)[8]) const {
    const uint8_t* b = stage + off + (lr >> 5) * (kTileC * 128) + (lr & 3) * 4;
    const int ch = (lr & 31) >> 2;
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = *reinterpret_cast<const float*>(b + swz(lc0 + k, ch));
  }
  __device__ __forceinline__ void col(int off, float (&t)[8]) const {
    const float4* p = reinterpret_cast<const float4*>(stage + off + lc0 * 4);
    const float4 a = p[0], c = p[1];
    t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w;
    t[4] = c.x; t[5] = c.y; t[6] = c.z; t[7] = c.w;
  }
  __device__ __forceinline__ void row(int off, float (&t)[8]) const {
    const float v = *reinterpret_cast<const float*>(stage + off + lr * 4);
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = v;
  }
  // f = sum_k ((g / d_k) % m_k) * s_k over g = r*FC + c (frames with gathered
  // leaves hold fewer than 2^31 elements)
  __device__ __forceinline__ void gather(int leaf, float (&t)[8]) const {
    const LeafDesc& G = P.leaves[leaf];
    const int r = r0 + lr;
    // every offset first, then the eight loads together (one memory latency,
    // not eight)
    uint32_t f[8];
    bool ok[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = c0 + lc0 + k;
      ok[k] = r < P.FR && c < P.FC;
      uint32_t g = (uint32_t)r * (uint32_t)P.FC + (uint32_t)c;
      if (G.shift) {
        // a tuple's field: other fields' points map outside it
        ok[k] = ok[k] && (int64_t)g >= G.shift;
        g = (uint32_t)((int64_t)g - G.shift);
      }
      f[k] = ok[k] ? digit_offset(G, g) : 0u;
      if (G.shift) ok[k] = ok[k] && (int64_t)f[k] < G.numel;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = ok[k] ? __ldg(G.ptr + f[k]) : 0.f;
  }
  // Extra output j: this thread's eight frame points, written where the
  // output's map sends them: rows of 32 contiguous bytes for the identity; a
  // transposed output gets 128-byte runs across the warp (lane = frame row);
  // any other permutation is evaluated digit by digit (frames with such
  // outputs hold fewer than 2^31 elements).
  __device__ __forceinline__ void xstore(int j, const float (&v)[8]) const {
    const XOutDesc& X = P.xout[j];
    if (xb) {
      // staged for the warp's TMA store: identity slices as [32 rows][8],
      // transposed ones as [8 rows][32] (lane = column of the output)
      uint8_t* b = xb + j * kXOutSliceBytes;
      if (X.cls == LEAF_IDENT) {
        float4* p = reinterpret_cast<float4*>(b + lr * 32);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) reinterpret_cast<float*>(b)[k * 32 + lr] = v[k];
      }
      return;
    }
    const int r = r0 + lr, c = c0 + lc0;
    if (r >= P.FR) return;
    if (X.cls == LEAF_IDENT) {
      float* op = X.ptr + (int64_t)r * P.FC + c;
      if ((P.FC & 3) == 0 && c + 8 <= P.FC) {
        reinterpret_cast<float4*>(op)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(op)[1] = make_float4(v[4], v[5], v[6], v[7]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (c + k < P.FC) op[k] = v[k];
      }
    } else if (X.cls == LEAF_TRANS) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (c + k < P.FC) X.ptr[(int64_t)(c + k) * P.FR + r] = v[k];
    } else {
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {
        if (c + k >= P.FC) break;
        const uint32_t g = (uint32_t)r * (uint32_t)P.FC + (uint32_t)(c + k);
        X.ptr[digit_offset(X, g)] = v[k];
      }
    }
  }
};

// ---- small groups: leaf reads straight from global memory -----------------------
// One thread's eight frame points (r0, c0 .. c0+7); lr = lc0 = 0 keep the
// select expressions of compiled programs valid (they test te.r0 + te.lr and
// te.c0 + te.lc0 + k).
struct DirectEnv {
  const GroupParams& P;
  int r0, lr, c0, lc0;

  __device__ __forceinline__ void ident_l(int l, float (&t)[8]) const {
    const float* p = P.leaves[l].ptr + (int64_t)r0 * P.FC + c0;
    if (c0 + 8 <= P.FC && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(p)), c = __ldg(reinterpret_cast<const float4*>(p) + 1);
      t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w;
      t[4] = c.x; t[5] = c.y; t[6] = c.z; t[7] = c.w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) t[k] = c0 + k < P.FC ? __ldg(p + k) : 0.f;
    }
  }
  // the leaf is the transposed value, [FC, FR]
  __device__ __forceinline__ void trans_l(int l, float (&t)[8]) const {
    const float* p = P.leaves[l].ptr + r0;
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = c0 + k < P.FC ? __ldg(p + (int64_t)(c0 + k) * P.FR) : 0.f;
  }
  __device__ __forceinline__ void col_l(int l, float (&t)[8]) const {
    const float* p = P.leaves[l].ptr + c0;
    if (c0 + 8 <= P.FC && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(p)), c = __ldg(reinterpret_cast<const float4*>(p) + 1);
      t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w;
      t[4] = c.x; t[5] = c.y; t[6] = c.z; t[7] = c.w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) t[k] = c0 + k < P.FC ? __ldg(p + k) : 0.f;
    }
  }
  __device__ __forceinline__ void row_l(int l, float (&t)[8]) const {
    const float v = __ldg(P.leaves[l].ptr + r0);
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = v;
  }
  // f = sum_k ((g / d_k) % m_k) * s_k over g = r*FC + c (small frames)
  __device__ __forceinline__ void gather(int leaf, float (&t)[8]) const {
    const LeafDesc& G = P.leaves[leaf];
    uint32_t f[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      f[k] = c0 + k < P.FC ? digit_offset(G, (uint32_t)r0 * (uint32_t)P.FC + (uint32_t)(c0 + k)) : 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = c0 + k < P.FC ? __ldg(G.ptr + f[k]) : 0.f;
  }
};

// Issues the TMA loads of one staged leaf for the tile at (r0, c0).
__device__ __forceinline__ void issue_leaf(const CUtensorMap* m, int cls, uint32_t dst, uint32_t bar, int r0, int c0) {
  if (cls == LEAF_IDENT) {
    tma_load_2d(dst, m, c0, r0, bar);
    tma_load_2d(dst + kTileR * 128, m, c0 + 32, r0, bar);
  } else if (cls == LEAF_TRANS) {
    tma_load_2d(dst, m, r0, c0, bar);
  } else if (cls == LEAF_COL) {
    tma_load_1d(dst, m, c0, bar);
  } else if (cls == LEAF_ROW) {
    tma_load_1d(dst, m, r0, bar);
  }
}

// ---- the interpreter as a program policy ---------------------------------------
struct LeafInfo {
  int32_t cls, stage_off, map_idx, pad;
};

// The program and the leaf table are copied to shared memory once per CTA:
// every thread reads them at every instruction.
struct SmemTables {
  VmInstr prog[kMaxProg];
  VmInstr epi[kMaxEpi];
  LeafInfo leaf[kMaxLeaves];
};

template <int D, int S>
struct InterpProg {
  using Tables = SmemTables;
  static constexpr int kMinBlocks = D <= 4 ? 2 : 1;

  __device__ static void load_tables(Tables& T, const GroupParams& P) {
    for (int i = threadIdx.x; i < P.nprog; i += blockDim.x) T.prog[i] = P.prog[i];
    for (int i = threadIdx.x; i < P.nepi; i += blockDim.x) T.epi[i] = P.epi[i];
    for (int i = threadIdx.x; i < P.nleaves; i += blockDim.x)
      T.leaf[i] = LeafInfo{P.leaves[i].cls, P.leaves[i].stage_off, P.leaves[i].map_idx, 0};
  }
  __device__ static void prefetch(const GroupParams& P, const Tables& T) {
    for (int j = 0; j < P.nleaves; ++j)
      if (T.leaf[j].cls != LEAF_GATHER) tma_prefetch(&P.maps[T.leaf[j].map_idx]);
  }
  __device__ static void issue(const GroupParams& P, const Tables& T, uint32_t st, uint32_t bar, int r0, int c0) {
    for (int j = 0; j < P.nleaves; ++j) {
      const LeafInfo L = T.leaf[j];
      if (L.cls != LEAF_GATHER) issue_leaf(&P.maps[L.map_idx], L.cls, st + L.stage_off, bar, r0, c0);
    }
  }
  struct Env {
    const TileEnv& te;
    const LeafInfo* leaf;
    __device__ __forceinline__ void load_leaf(int arg, float (&t)[8]) const {
      const LeafInfo L = leaf[arg];
      if (L.cls == LEAF_IDENT) te.ident(L.stage_off, t);
      else if (L.cls == LEAF_TRANS) te.trans(L.stage_off, t);
      else if (L.cls == LEAF_COL) te.col(L.stage_off, t);
      else if (L.cls == LEAF_ROW) te.row(L.stage_off, t);
      else te.gather(arg, t);
    }
    __device__ __forceinline__ void load_acc(float (&t)[8]) const {
#pragma unroll
      for (int k = 0; k < 8; ++k) t[k] = 0.f;
    }
  };
  __device__ __forceinline__ static void run(const TileEnv& te, const Tables& T, const GroupParams& P, float (&o)[8]) {
    Machine<D, S, 8> M;
    Env env{te, T.leaf};
    M.run(T.prog, P.nprog, env);
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = M.TOP[k];
  }
  // reduce epilogue on the reduced value of row r
  __device__ static float epi(const GroupParams& P, const Tables& T, int r, float acc) {
    if (P.nepi == 0) return acc;
    struct EpiEnv {
      const GroupParams& P;
      int r;
      float a;
      __device__ __forceinline__ void load_leaf(int arg, float (&t)[1]) const { t[0] = __ldg(P.epi_leaf[arg] + r); }
      __device__ __forceinline__ void load_acc(float (&t)[1]) const { t[0] = a; }
    } env{P, r, acc};
    Machine<D, S, 1> E;
    E.run(T.epi, P.nepi, env);
    return E.TOP[0];
  }
};

// ---- pipeline pieces ----------------------------------------------------------------
struct Ring {
  uint8_t* base;        // generic pointer to stage 0
  uint32_t base_s;      // shared address of stage 0
  uint32_t full_s, empty_s;
};

__device__ __forceinline__ Ring setup_ring(uint8_t* smem) {
  Ring R;
  R.full_s = smem_u32(smem);
  R.empty_s = R.full_s + 8 * kMaxStages;
  R.base = smem + 1024;
  R.base_s = smem_u32(R.base);
  return R;
}

__device__ __forceinline__ void init_barriers(const Ring& R, int NS) {
  for (int s = 0; s < NS; ++s) {
    mbar_init(R.full_s + 8 * s, 1);
    mbar_init(R.empty_s + 8 * s, kConsumerWarps);
  }
  fence_mbar_init();
}

// Named barrier 1 over the consumer warps, returning the OR of `pred`.
__device__ __forceinline__ bool consumer_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kConsumers)
      : "memory");
  return r != 0;
}

// Linear tile index -> (tile row, tile col): row-major, or column-major inside
// bands of `band` tile rows.
__device__ __forceinline__ void tile_coords(int t, int ntr, int ntc, int band, int& tr, int& tc) {
  if (band <= 0) {
    tr = t / ntc;
    tc = t % ntc;
    return;
  }
  const int per = band * ntc;
  const int b = t / per, local = t - b * per;
  const int rows = min(band, ntr - b * band);
  tr = b * band + local % rows;
  tc = local / rows;
}

struct RedTiles {   // units (row strip, column split), then the split's tiles
  int u, step, nunits, nsplit, tps, ntc;
  int tc, tc_end, strip;
  bool started;
  __device__ __forceinline__ bool next(int& tr, int& tcol) {
    while (!started || tc >= tc_end) {
      if (started) u += step;
      started = true;
      if (u >= nunits) return false;
      strip = u / nsplit;
      tc = (u % nsplit) * tps;
      tc_end = min(ntc, tc + tps);
    }
    tr = strip;
    tcol = tc++;
    return true;
  }
};

// Elementwise groups claim their tiles dynamically from the group's claim
// counter (P.sched, 64 bits) with atomic adds.  SMs do not stream at the same
// rate (with a fixed split of the tiles the slowest CTAs finished several
// microseconds after the rest, the memory system half idle meanwhile);
// claiming keeps every CTA busy until the tiles run out.  Each producer's
// first tile is fixed (no launch-time rush on the counter); later tiles are
// claimed, one claim ahead.  A launch makes exactly as many claims as it has
// tiles (each producer with a valid first tile claims until one claim fails),
// so the counter never needs resetting: claim c is tile first + c mod ntiles
// of its launch.  (A launch that gave up on a bounded wait leaves the count
// off; the host clears the counter when it reports the timeout.)  Producer p
// fills the stages i with i % 2 == p (the ring depth is even, so each owns
// half of the slots); each stage carries its tile row and column (-1: the
// producer has no more tiles).
__device__ __forceinline__ int claim_unit(unsigned long long* ctr, int first, int nunits) {
  const unsigned long long c = atomicAdd(ctr, 1ull);
  return first + (int)(c % (unsigned long long)nunits);
}

struct EwUnits {   // one tile per unit, in the tile walk's order
  int nunits, ntr, ntc, band;
  __device__ __forceinline__ int tiles(int) const { return 1; }
  __device__ __forceinline__ void tile(int u, int, int& tr, int& tc) const { tile_coords(u, ntr, ntc, band, tr, tc); }
};

// An elementwise producer (one thread): claims tiles until they run out,
// issues the TMA loads of every staged leaf of each into its stages (a thread
// takes a few hundred ns to wait for a stage, arm it and issue its copies:
// two producers keep more loads in flight), then marks its last stage.  The
// next claim is in flight while the current tile is issued.  On a timeout it
// waits for its loads still in flight.
template <class Prog, class Units>
__device__ __forceinline__ void ew_producer(const GroupParams& P, const typename Prog::Tables& T, const Ring& R,
                                            int2* info, const Units U, volatile int* abort_flag, int par) {
  if (P.inject) return;   // failure injection: consumers wait for loads that never come
  Prog::prefetch(P, T);
  const int NS = P.nstages;
  int i = par;
  bool ok = true;
  // the first tile of each producer is fixed (no launch-time rush on the
  // counter); claims number the tiles after those
  const int first = 2 * (int)gridDim.x;
  int next = 2 * (int)blockIdx.x + par;
  for (;;) {
    const int u = next;
    if (u >= U.nunits) break;
    next = claim_unit(P.sched, first, U.nunits);
    const int nt = U.tiles(u);
    for (int k = 0; k < nt && ok; ++k, i += kProducerWarps) {
      const int s = i % NS;
      if (i >= NS && !wait_or_abort(R.empty_s + 8 * s, ((i / NS) & 1) ^ 1, P.wait_limit_ns, abort_flag)) {
        ok = false;
        break;
      }
      int tr, tc;
      U.tile(u, k, tr, tc);
      info[s] = make_int2(tr, tc);
      const uint32_t bar = R.full_s + 8 * s;
      mbar_expect_tx(bar, P.tx_bytes);
      Prog::issue(P, T, R.base_s + s * P.stage_bytes, bar, tr * kTileR, tc * kTileC);
    }
    if (!ok) break;
  }
  if (ok) {
    const int s = i % NS;
    if (i >= NS && !wait_or_abort(R.empty_s + 8 * s, ((i / NS) & 1) ^ 1, P.wait_limit_ns, abort_flag)) {
      ok = false;
    } else {
      info[s] = make_int2(-1, 0);
      mbar_arrive(R.full_s + 8 * s);
    }
  }
  if (!ok) {
    *abort_flag = 1;
    set_error(P.err, DEVERR_TIMEOUT);
    const int64_t drain = P.wait_limit_ns > kDrainLimitNs ? P.wait_limit_ns : kDrainLimitNs;
    for (int k = i - NS < 0 ? 0 : i - NS; k < i; ++k)
      if (k % kProducerWarps == par) mbar_wait(R.full_s + 8 * (k % NS), (k / NS) & 1, drain);
  }
}

// A reduce producer: one thread issues the TMA loads of every staged leaf for
// the tiles i = par, par + kProducerWarps, ... into the ring (a thread takes a few
// hundred ns to wait for a stage, arm it and issue its copies: two producers
// keep more loads in flight); on a timeout it waits for its loads still in
// flight.  With at least two stages, each producer's previous wait ensures the
// parity it waits for belongs to the current use of the stage.
template <class Prog, class Tiles>
__device__ __forceinline__ void producer_loop(const GroupParams& P, const typename Prog::Tables& T, const Ring& R,
                                              Tiles tiles, volatile int* abort_flag, int par) {
  if (P.inject) return;   // failure injection: consumers wait for loads that never come
  Prog::prefetch(P, T);
  const int NS = P.nstages;
  int i = 0, tr, tc;
  bool ok = true;
  while (tiles.next(tr, tc)) {
    if (i % kProducerWarps != par) {
      ++i;
      continue;
    }
    const int s = i % NS;
    if (i >= NS && !wait_or_abort(R.empty_s + 8 * s, ((i / NS) & 1) ^ 1, P.wait_limit_ns, abort_flag)) {
      ok = false;
      break;
    }
    const uint32_t bar = R.full_s + 8 * s;
    mbar_expect_tx(bar, P.tx_bytes);
    Prog::issue(P, T, R.base_s + s * P.stage_bytes, bar, tr * kTileR, tc * kTileC);
    ++i;
  }
  if (!ok) {
    *abort_flag = 1;
    set_error(P.err, DEVERR_TIMEOUT);
    const int64_t drain = P.wait_limit_ns > kDrainLimitNs ? P.wait_limit_ns : kDrainLimitNs;
    for (int k = i - NS < 0 ? 0 : i - NS; k < i; ++k)
      if (k % kProducerWarps == par) mbar_wait(R.full_s + 8 * (k % NS), (k / NS) & 1, drain);
  }
}

// ---------------------------------------------------------------------------------
// K1 body: elementwise / broadcast / injective group.
template <class Prog>
__device__ __forceinline__ void ew_body(const GroupParams& P) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ typename Prog::Tables T;
  __shared__ int2 info[kMaxStages];
  uint8_t* smem = align1024(smem_raw);
  const Ring R = setup_ring(smem);
  uint8_t* outbuf = R.base + P.nstages * P.stage_bytes;
  uint8_t* xbuf = outbuf + 3 * kOutBufBytes;   // [3][nxout][8 warps][32 x 8 floats]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Prog::load_tables(T, P);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    init_barriers(R, P.nstages);
    if (P.out_tma) tma_prefetch(&P.maps[kMaxStaged]);
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();   // the previous grid's writes are visible from here on

  if (warp >= kConsumerWarps) {
    if (lane == 0)
      ew_producer<Prog>(P, T, R, info, EwUnits{P.ntiles, P.ntr, P.ntc, P.band}, &abort_flag,
                          warp - kConsumerWarps);
  } else {
    const int NS = P.nstages;
    const int lr = lane, lc0 = warp * 8;
    const bool vec_store = (P.FC & 3) == 0 && (reinterpret_cast<uintptr_t>(P.out) & 15) == 0;
    float o[8];
    static_assert(kProducerWarps == 2, "two producers, owning the even and the odd stages");
    bool fin0 = false, fin1 = false;   // producers whose last stage has been seen
    for (int i = 0; !(fin0 && fin1); ++i) {
      if (i & 1 ? fin1 : fin0) continue;
      const int s = i % NS;
      const bool got = wait_or_abort(R.full_s + 8 * s, (i / NS) & 1, P.wait_limit_ns, &abort_flag);
      const int2 inf = got ? info[s] : make_int2(0, 0);
      if (inf.x < 0) {
        // that producer has no more tiles (every warp that waited reads the
        // same stage).  With the CTA-wide store every warp takes exactly one
        // barrier per stage it waits for, this one included, so that a warp
        // that gave up on it meets the others there
        if (P.out_tma == 1 && consumer_bar_or(false)) break;
        if (i & 1) fin1 = true;
        else fin0 = true;
        continue;
      }
      const int r0 = inf.x * kTileR, c0 = inf.y * kTileC;   // the tile's row and column tiles
      uint8_t* ob = outbuf + (i % 3) * kOutBufBytes;
      if (got) {
        const TileEnv te{P, R.base + s * P.stage_bytes, lr, lc0, r0, c0,
                         P.xout_tma ? xbuf + ((i % 3) * P.nxout * 8 + warp) * (kTileR * 32) : nullptr};
        Prog::run(te, T, P, o);
        if (P.out_tma == 1) {
          uint8_t* b = ob + (lc0 >> 5) * (kTileR * 128);
          const int j0 = (lc0 & 31) >> 2;
          *reinterpret_cast<float4*>(b + swz(lr, j0)) = make_float4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<float4*>(b + swz(lr, j0 + 1)) = make_float4(o[4], o[5], o[6], o[7]);
        } else if (P.out_tma == 2) {
          // this warp's 32 x 8 slice, row-major, stored by its own lane 0;
          // lanes 4-7 of every eight write their rows' halves in the other
          // order, so that each eight lanes' 16-byte stores cover all banks
          float4* b = reinterpret_cast<float4*>(ob + warp * (kTileR * 32) + lr * 32);
          const float4 lo = make_float4(o[0], o[1], o[2], o[3]), hi = make_float4(o[4], o[5], o[6], o[7]);
          const int h = (lr >> 2) & 1;
          b[h] = h ? hi : lo;
          b[h ^ 1] = h ? lo : hi;
        } else {
          // each lane writes 32 contiguous bytes of its row: whole sectors
          const int r = r0 + lr, c = c0 + lc0;
          if (r < P.FR) {
            float* op = P.out + (int64_t)r * P.FC + c;
            if (vec_store && c + 8 <= P.FC) {
              reinterpret_cast<float4*>(op)[0] = make_float4(o[0], o[1], o[2], o[3]);
              reinterpret_cast<float4*>(op)[1] = make_float4(o[4], o[5], o[6], o[7]);
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                if (c + k < P.FC) op[k] = o[k];
            }
          }
        }
      } else {
        abort_flag = 1;
        set_error(P.err, DEVERR_TIMEOUT);
      }
      if (P.out_tma == 2) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(R.empty_s + 8 * s);
          if (got && c0 + lc0 < P.FC) {
            tma_store_2d(&P.maps[kMaxStaged], c0 + lc0, r0, smem_u32(ob + warp * (kTileR * 32)));
            if (P.xout_tma) {
              const uint8_t* xw = xbuf + ((i % 3) * P.nxout * 8 + warp) * (kTileR * 32);
              for (int j = 0; j < P.nxout; ++j) {
                if (P.xout[j].cls == LEAF_IDENT)
                  tma_store_2d(&P.xmaps[j], c0 + lc0, r0, smem_u32(xw + j * kXOutSliceBytes));
                else
                  tma_store_2d(&P.xmaps[j], r0, c0 + lc0, smem_u32(xw + j * kXOutSliceBytes));
              }
            }
            bulk_commit();
            bulk_wait_read<1>();
          }
        }
        __syncwarp();
        if (!got) break;
        continue;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(R.empty_s + 8 * s);
      if (P.out_tma == 1) {
        // every consumer warp reaches this barrier once per tile it waited
        // for: one that gave up leaves together with the others
        fence_proxy_async_smem();
        if (consumer_bar_or(!got)) break;
        if (threadIdx.x == 0) {
          const uint32_t src = smem_u32(ob);
          tma_store_2d(&P.maps[kMaxStaged], c0, r0, src);
          if (c0 + 32 < P.FC) tma_store_2d(&P.maps[kMaxStaged], c0 + 32, r0, src + kTileR * 128);
          bulk_commit();
          bulk_wait_read<1>();
        }
      } else if (!got) {
        break;
      }
    }
    if (P.out_tma == 1 && threadIdx.x == 0) bulk_wait<0>();
    if (P.out_tma == 2 && lane == 0) bulk_wait<0>();
  }
}

// A consumer warp of a reduce CTA, once the count of a split unit of `strip` has
// arrived (`old`: the counter before its increment, lane 0): the unit that
// counted last acquires the other
// units' partials (their release increments precede its own in the counter's
// order), sums them in split order, loads issued eight at a time, and writes
// the epilogue's result.
template <class Prog>
__device__ __forceinline__ void reduce_finish(const GroupParams& P, const typename Prog::Tables& T, int strip,
                                              int old, bool is_sum) {
  const int lane = threadIdx.x & 31;
  const bool last = __shfl_sync(0xffffffffu, old, 0) == P.nsplit - 1;
  if (!last) return;
  fence_acq_rel_gpu();
  __syncwarp();
  const int r = strip * kTileR + lane;
  float p = is_sum ? 0.f : neg_inf();
  if (r < P.FR) {
    for (int q0 = 0; q0 < P.nsplit; q0 += 8) {
      float x[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        x[k] = q0 + k < P.nsplit ? __ldcg(P.scratch + (int64_t)(q0 + k) * P.FR + r) : (is_sum ? 0.f : neg_inf());
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (q0 + k < P.nsplit) p = is_sum ? __fadd_rn(p, x[k]) : fmaxf(p, x[k]);
    }
    P.out[r] = Prog::epi(P, T, r, p);
  }
  if (lane == 0) P.counters[strip] = 0;
}

// ---------------------------------------------------------------------------------
// K2 body: group ending in a row reduction over the frame's last axis, with an
// optional elementwise epilogue on the reduced vector.  Work units are
// (32-row strip, run of column tiles); a unit writes its partial row values
// to scratch and the last unit of a strip to arrive combines them in split
// order, so the result does not depend on scheduling.
template <class Prog>
__device__ __forceinline__ void reduce_body(const GroupParams& P) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ typename Prog::Tables T;
  uint8_t* smem = align1024(smem_raw);
  const Ring R = setup_ring(smem);
  float* red = reinterpret_cast<float*>(R.base + P.nstages * P.stage_bytes);   // [2][8 warps][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Prog::load_tables(T, P);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    init_barriers(R, P.nstages);
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();   // the previous grid's writes are visible from here on

  if (warp >= kConsumerWarps) {
    if (lane == 0)
      producer_loop<Prog>(P, T, R,
                          RedTiles{(int)blockIdx.x, (int)gridDim.x, P.nunits, P.nsplit, P.tiles_per_split, P.ntc, 0, 0,
                                   0, false},
                          &abort_flag, warp - kConsumerWarps);
    return;
  }

  const int NS = P.nstages;
  const int lr = lane, lc0 = warp * 8;
  const bool is_sum = P.red_op == RED_SUM;
  float o[8];
  int i = 0, k_unit = 0;
  bool dead = false;
  int pend_strip = -1, pend_old = 0;   // this warp's split unit whose count is in flight
  for (int u = blockIdx.x; u < P.nunits; u += gridDim.x, ++k_unit) {
    const int strip = u / P.nsplit, sp = u % P.nsplit;
    const int tcb = sp * P.tiles_per_split;
    const int tce = min(P.ntc, tcb + P.tiles_per_split);
    const int r0 = strip * kTileR;
    float acc = is_sum ? 0.f : neg_inf();
    for (int tc = tcb; tc < tce; ++tc, ++i) {
      const int s = i % NS;
      const int c0 = tc * kTileC;
      const bool got = !dead && wait_or_abort(R.full_s + 8 * s, (i / NS) & 1, P.wait_limit_ns, &abort_flag);
      if (got) {
        const TileEnv te{P, R.base + s * P.stage_bytes, lr, lc0, r0, c0};
        Prog::run(te, T, P, o);
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const bool in = c0 + lc0 + k < P.FC;
          v[k] = in ? o[k] : (is_sum ? 0.f : neg_inf());
        }
        if (is_sum) {
          acc = __fadd_rn(acc, __fadd_rn(__fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3])),
                                         __fadd_rn(__fadd_rn(v[4], v[5]), __fadd_rn(v[6], v[7]))));
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) acc = fmaxf(acc, v[k]);
        }
      } else if (!dead) {
        dead = true;
        abort_flag = 1;
        set_error(P.err, DEVERR_TIMEOUT);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(R.empty_s + 8 * s);
    }
    float* rb = red + (k_unit & 1) * (kConsumerWarps * 32);
    rb[warp * 32 + lane] = acc;
    if (consumer_bar_or(dead)) break;
    // the unit's combine falls to the warps in turn: publishing partials
    // holds the publishing warp until its stores are acknowledged, and one
    // warp in eight units is a stall the ring absorbs
    if (warp == k_unit % kConsumerWarps) {
      float p = rb[lane];
      for (int w = 1; w < kConsumerWarps; ++w) p = is_sum ? __fadd_rn(p, rb[w * 32 + lane]) : fmaxf(p, rb[w * 32 + lane]);
      const int r = r0 + lane;
      if (P.nsplit > 1) {
        // this warp's previous split unit's count has arrived by now:
        // finish its strip if it counted last; then publish this unit's
        // partials with a release increment whose old value is read only at
        // this warp's next combine
        if (pend_strip >= 0) reduce_finish<Prog>(P, T, pend_strip, pend_old, is_sum);
        if (r < P.FR) P.scratch[(int64_t)sp * P.FR + r] = p;
        __syncwarp();
        if (lane == 0) pend_old = atom_add_release_gpu(&P.counters[strip], 1);   // compared at the next end
        pend_strip = strip;
      } else if (r < P.FR) {
        P.out[r] = Prog::epi(P, T, r, p);
      }
    }
  }
  if (pend_strip >= 0 && !dead) reduce_finish<Prog>(P, T, pend_strip, pend_old, is_sum);
}

// ---------------------------------------------------------------------------------
// The direct kernel: no shared-memory ring, leaves read straight from global
// memory.  It runs small groups (a couple of MB of leaves and output at most,
// rows of at most 1024 columns), elementwise or ending in a row reduction,
// where the pipelined kernels' set-up (barriers, descriptor fetches, split
// combines) would cost several round trips to memory; and larger row
// reductions whose leaves are all read row by row (the frame's own layout,
// vectors over its rows or columns), where each warp's contiguous run of a
// row keeps the memory system's pages busier than the pipeline's 32-row
// tiles (the CTA scheduler also spreads the short CTAs over the SMs as they
// free up).  One warp per frame row segment (P.seg warps per row, each
// P.seg_cols columns), eight consecutive frame columns per lane and pass.
// A reduction folds each lane's values in order, then the lanes in a fixed
// butterfly, then the row's segments in order; one lane applies the
// epilogue.
template <class Prog, bool kSeg>
__device__ __forceinline__ void small_body(const GroupParams& P) {
  // the segments' partials (kSeg: launched with this much dynamic shared
  // memory; a one-segment launch has neither it nor the barrier, and its
  // warps without a row leave at once: measured 0.6 us less per run on the
  // two-group RNNLM chain than the segmented body with one segment)
  extern __shared__ float part[];
  pdl_launch_dependents();
  pdl_wait();   // the previous grid's writes are visible from here on
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wid = blockIdx.x * (kSmallThreads / 32) + warp;
  int r = wid, sg = 0, c_begin = 0, c_end = P.FC;
  if constexpr (kSeg) {
    const int S = P.seg;   // a power of two dividing the CTA's warps: a row's segments share a CTA
    r = wid / S;
    sg = wid - r * S;
    c_begin = sg * P.seg_cols;
    c_end = min(P.FC, c_begin + P.seg_cols);
  } else if (r >= P.FR) {
    return;
  }
  const bool red = P.red_op != RED_NONE, is_sum = P.red_op == RED_SUM;
  const float init = is_sum ? 0.f : neg_inf();
  float acc = init;
  if (r < P.FR) {
#pragma unroll 2
    for (int c = c_begin + lane * 8; c < c_end; c += 32 * 8) {
      const DirectEnv te{P, r, 0, c, 0};
      float o[8];
      Prog::run_direct(te, o);
      if (red) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = c + k < P.FC ? o[k] : init;
        if (is_sum) {
          acc = __fadd_rn(acc, __fadd_rn(__fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3])),
                                         __fadd_rn(__fadd_rn(v[4], v[5]), __fadd_rn(v[6], v[7]))));
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) acc = fmaxf(acc, v[k]);
        }
      } else {
        float* op = P.out + (int64_t)r * P.FC + c;
        if (c + 8 <= P.FC && (reinterpret_cast<uintptr_t>(op) & 15) == 0) {
          reinterpret_cast<float4*>(op)[0] = make_float4(o[0], o[1], o[2], o[3]);
          reinterpret_cast<float4*>(op)[1] = make_float4(o[4], o[5], o[6], o[7]);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (c + k < P.FC) op[k] = o[k];
        }
      }
    }
  }
  if (!red) return;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, acc, d);
    acc = is_sum ? __fadd_rn(acc, x) : fmaxf(acc, x);
  }
  if constexpr (kSeg) {
    // every warp of the CTA reaches this barrier
    if (lane == 0) part[warp] = acc;
    __syncthreads();
    if (sg != 0) return;
    for (int k = 1; k < P.seg; ++k) acc = is_sum ? __fadd_rn(acc, part[warp + k]) : fmaxf(acc, part[warp + k]);
  }
  const typename Prog::Tables T{};
  if (lane == 0 && r < P.FR) P.out[r] = Prog::epi(P, T, r, acc);
}

}  // namespace fg
