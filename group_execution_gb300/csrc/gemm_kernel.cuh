// GEMM-epilogue group kernel (K3): D = A * B on the 5th-generation tensor
// cores with the group's elementwise tail applied to the accumulator before
// it ever reaches global memory (TVM "Operator Fusion", Fusion rules, phase
// 0: an out-elementwise-fusable operator such as matmul fuses with its
// elementwise successors; TAG's sufficient-factor gradient G = U^T V is the
// workload).
//
// Persistent: CTAs run in pairs (a 2-CTA cluster) on the SMs of one TPC, and
// a pair walks 256 x 256 output tiles.  Each CTA stages half of the tile's A
// rows and half of its B columns, two 64-deep K blocks (64 KB) per ring slot,
// each operand half in one TMA copy where the layout allows; the even CTA
// issues 2-SM tcgen05.mma instructions (cta_group::2) that read both CTAs'
// halves and leave each CTA's 128 accumulator rows in its own TMEM.  Warp
// roles, in each CTA:
//   warp 0  TMA producer of the bf16 operand halves; every load completes on
//           the even CTA's stage barrier,
//   warp 1  allocates TMEM (2 x 256 columns: double-buffered accumulator,
//           jointly with the peer) and, in the even CTA, issues the MMAs from
//           one thread,
//   warp 2  TMA producer of the epilogue leaves, 128 x 32 chunk by chunk,
//   warps 3-6 epilogue: each thread owns one accumulator row (TMEM lane),
//           reads 32 columns per chunk with tcgen05.ld, evaluates the
//           epilogue program eight values at a time and stages the result
//           for a TMA store.
// The epilogue of tile i overlaps the MMAs of tile i+1.  Every wait is
// bounded; on expiry the CTA records the error, drains its copies, frees its
// TMEM and returns.
#pragma once
#include "fg_device.cuh"

namespace fg {

constexpr int kGemmThreads = kGemmWarps * 32;
constexpr int kGemmABytes = kGemmM * kGemmK * 2;    // 16 KB: this CTA's 128 rows of one A block
constexpr int kGemmOutBytes = kGemmM * kGemmChunk * 4;   // 16 KB
constexpr int kGemmChunks = kGemmN / kGemmChunk;    // 8

// Leaf reads for one epilogue thread: accumulator row rr of the tile, eight
// columns starting at q8 inside the current 32-column chunk.
struct GemmEnv {
  const GemmParams& P;
  const uint8_t* stage;
  int rr, r0, cc0, q8;

  __device__ __forceinline__ static int swz(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }
  __device__ __forceinline__ void ident(int off, float (&t)[8]) const {
    const uint8_t* b = stage + off;
    const float4 a = *reinterpret_cast<const float4*>(b + swz(rr, q8 >> 2));
    const float4 c = *reinterpret_cast<const float4*>(b + swz(rr, (q8 >> 2) + 1));
    t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w;
    t[4] = c.x; t[5] = c.y; t[6] = c.z; t[7] = c.w;
  }
  // four 32 x 32 boxes, box b holding tile rows 32b..32b+31 transposed
  __device__ __forceinline__ void trans(int off, float (&t)[8]) const {
    const uint8_t* b = stage + off + (rr >> 5) * 4096 + (rr & 3) * 4;
    const int ch = (rr & 31) >> 2;
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = *reinterpret_cast<const float*>(b + swz(q8 + k, ch));
  }
  __device__ __forceinline__ void col(int off, float (&t)[8]) const {
    const float4* p = reinterpret_cast<const float4*>(stage + off + q8 * 4);
    const float4 a = p[0], c = p[1];
    t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w;
    t[4] = c.x; t[5] = c.y; t[6] = c.z; t[7] = c.w;
  }
  __device__ __forceinline__ void row(int off, float (&t)[8]) const {
    const float v = *reinterpret_cast<const float*>(stage + off + rr * 4);
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = v;
  }
  __device__ __forceinline__ void gather(int leaf, float (&t)[8]) const {
    const LeafDesc& G = P.leaves[leaf];
    const int r = r0 + rr;
#pragma unroll 1
    for (int k = 0; k < 8; ++k) {
      const int c = cc0 + q8 + k;
      float v = 0.f;
      if (r < P.M && c < P.N) {
        const uint32_t g = (uint32_t)r * (uint32_t)P.N + (uint32_t)c;
        uint32_t f = 0;
        for (int q = 0; q < G.nterms; ++q) f += ((g / (uint32_t)G.d[q]) % (uint32_t)G.m[q]) * (uint32_t)G.s[q];
        v = __ldg(G.ptr + f);
      }
      t[k] = v;
    }
  }
};

// TMA loads of one staged epilogue leaf for rows r0..r0+127, columns
// cc0..cc0+31.
__device__ __forceinline__ void gemm_issue_leaf(const CUtensorMap* m, int cls, uint32_t dst, uint32_t bar, int r0,
                                                int cc0) {
  // a tile's leaf boxes are read once: they leave L2 first
  const uint64_t once = l2_evict_first();
  if (cls == LEAF_IDENT) {
    tma_load_2d_hint(dst, m, cc0, r0, bar, once);
  } else if (cls == LEAF_TRANS) {
#pragma unroll
    for (int b = 0; b < 4; ++b) tma_load_2d_hint(dst + b * 4096, m, r0 + 32 * b, cc0, bar, once);
  } else if (cls == LEAF_COL) {
    tma_load_1d(dst, m, cc0, bar);
  } else if (cls == LEAF_ROW) {
    tma_load_1d(dst, m, r0, bar);
  }
}

// The interpreted epilogue.
template <int D, int S>
struct InterpGemmEpi {
  __device__ static void prefetch(const GemmParams& P) {
    for (int j = 0; j < P.nleaves; ++j)
      if (P.leaves[j].cls != LEAF_GATHER) tma_prefetch(&P.maps[P.leaves[j].map_idx]);
  }
  __device__ static void issue(const GemmParams& P, uint32_t st, uint32_t bar, int r0, int cc0) {
    for (int j = 0; j < P.nleaves; ++j) {
      const LeafDesc& L = P.leaves[j];
      if (L.cls != LEAF_GATHER) gemm_issue_leaf(&P.maps[L.map_idx], L.cls, st + L.stage_off, bar, r0, cc0);
    }
  }
  struct Env {
    const GemmEnv& ge;
    const float (&acc)[8];
    __device__ __forceinline__ void load_leaf(int arg, float (&t)[8]) const {
      const LeafDesc& L = ge.P.leaves[arg];
      if (L.cls == LEAF_IDENT) ge.ident(L.stage_off, t);
      else if (L.cls == LEAF_TRANS) ge.trans(L.stage_off, t);
      else if (L.cls == LEAF_COL) ge.col(L.stage_off, t);
      else if (L.cls == LEAF_ROW) ge.row(L.stage_off, t);
      else ge.gather(arg, t);
    }
    __device__ __forceinline__ void load_acc(float (&t)[8]) const {
#pragma unroll
      for (int k = 0; k < 8; ++k) t[k] = acc[k];
    }
  };
  __device__ __forceinline__ static void run(const GemmEnv& ge, const float (&acc)[8], float (&o)[8]) {
    Machine<D, S, 8> M;
    Env env{ge, acc};
    M.run(ge.P.prog, ge.P.nprog, env);
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = M.TOP[k];
  }
};

__device__ __forceinline__ bool gemm_wait(uint32_t bar, uint32_t parity, int64_t limit, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if ((int64_t)(global_ns() - t0) > limit) return false;
  }
  return true;
}

// One item of a pair's work list: a whole tile unit, or one K piece (ring
// slots [sl0, sl1)) of a unit of the split last round.
struct GemmItem {
  int unit, piece, sl0, sl1, q;   // piece = -1 for a whole unit; q = index among all pieces
};
__device__ __forceinline__ GemmItem gemm_item(const GemmParams& P, int idx, int nslots) {
  GemmItem w;
  if (idx < P.nfull) {
    w.unit = idx;
    w.piece = -1;
    w.sl0 = 0;
    w.sl1 = nslots;
    w.q = -1;
  } else {
    w.q = idx - P.nfull;
    w.unit = P.nfull + w.q / P.split;
    w.piece = w.q % P.split;
    w.sl0 = w.piece * nslots / P.split;
    w.sl1 = (w.piece + 1) * nslots / P.split;
  }
  return w;
}

// CL = 2: a CTA pair per 256 x 256 tile (cta_group::2), each CTA holding
// half of A's rows and half of B's columns.
template <class Epi, int CL>
__device__ __forceinline__ void gemm_body(const GemmParams& P) {
  static_assert(CL == 2, "the kernel runs CTA pairs");
  constexpr int kBCols = kGemmN / CL;                              // B columns staged per CTA
  constexpr int kHalfA = kGemmKB * kGemmABytes;                    // 32 KB: 128 rows x 2 K blocks
  constexpr int kStageBytes = kHalfA + kGemmKB * kBCols * kGemmK * 2;   // 64 KB per CTA
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_slot;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // barriers: full[16] empty[16] tfull[2] tempty[2] efull[8] eempty[8] done
  const uint32_t bars = smem_u32(smem);
  const uint32_t full0 = bars, empty0 = bars + 128, tfull0 = bars + 256, tempty0 = bars + 272;
  const uint32_t efull0 = bars + 288, eempty0 = bars + 352, done_bar = bars + 416;
  uint8_t* opnd = smem + 1024;
  const int NS = P.nstages, NE = P.n_epi_bufs;
  uint8_t* ebuf = opnd + NS * kStageBytes;
  uint8_t* obuf = ebuf + NE * P.epi_stage_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool staged = P.epi_tx_bytes > 0;
  const int nslots = (P.nkb + kGemmKB - 1) / kGemmKB;             // ring slots per tile

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  // tile sequence: units of CL vertically adjacent 128-row tiles
  const int ncl = gridDim.x / CL, cl = blockIdx.x / CL;
  const int npm = (P.ntm + CL - 1) / CL, nunits = npm * P.ntn;
  const int nitems = P.nfull + (nunits - P.nfull) * P.split;
  auto tile_of = [&](int u, int& m0, int& n0) {
    m0 = ((u / P.ntn) * CL + (int)rank) * kGemmM;
    n0 = (u % P.ntn) * kGemmN;
  };
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 4 * CL);   // every epilogue warp of the pair
    }
    for (int e = 0; e < NE; ++e) {
      mbar_init(efull0 + 8 * e, 1);
      mbar_init(eempty0 + 8 * e, 4);
    }
    mbar_init(done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc<CL>(smem_u32(&tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int64_t limit = P.wait_limit_ns;
  const int64_t drain = limit > kDrainLimitNs ? limit : kDrainLimitNs;

  if (warp == 0) {
    // ---- operand producer ----
    // Ring slot layouts (per CTA), each 128-byte row 128B-swizzled:
    //   K-major operand:  [K block][128 rows][64 K]        (16 KB per K block)
    //   MN-major operand: [64-wide group][128 K rows][64]  (16 KB per group)
    if (lane == 0 && !P.inject) {
      tma_prefetch(&P.mapA);
      tma_prefetch(&P.mapB);
      const uint64_t keep = l2_evict_last();   // every operand tile is read by several tiles
      int it = 0;
      bool ok = true;
      for (int x = cl; x < nitems && ok; x += ncl) {
        const GemmItem w = gemm_item(P, x, nslots);
        int m0, n0;
        tile_of(w.unit, m0, n0);
        const int nb = n0 + (int)rank * kBCols;
        for (int sl = w.sl0; sl < w.sl1; ++sl, ++it) {
          const int s = it % NS;
          if (it >= NS && !gemm_wait(empty0 + 8 * s, ((it / NS) & 1) ^ 1, limit, &abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t a = smem_u32(opnd + s * kStageBytes), b = a + kHalfA;
          const int k0 = sl * kGemmKB * kGemmK;
          // both CTAs' halves are counted on the even CTA's barrier, which
          // the even CTA alone arms with the whole slot's bytes (blocks past
          // K arrive zero-filled and count in full)
          const uint32_t cbar = cluster_addr(full0 + 8 * s, 0);
          if (leader) mbar_expect_tx(full0 + 8 * s, CL * kStageBytes);
          if (P.a_mn) {
            if (P.a_3d) {
              tma_load_3d_pair(a, &P.mapA, 0, k0, m0 / 64, cbar, keep);
            } else {
#pragma unroll
              for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                  tma_load_2d_pair(a + g * 16384 + j * 8192, &P.mapA, m0 + 64 * g, k0 + 64 * j, cbar, keep);
            }
          } else if (P.a_3d) {
            tma_load_3d_pair(a, &P.mapA, 0, m0, k0 / 64, cbar, keep);
          } else {
#pragma unroll
            for (int j = 0; j < kGemmKB; ++j) tma_load_2d_pair(a + j * 16384, &P.mapA, k0 + 64 * j, m0, cbar, keep);
          }
          if (P.b_mn) {
            if (P.b_3d) {
              tma_load_3d_pair(b, &P.mapB, 0, k0, nb / 64, cbar, keep);
            } else {
#pragma unroll
              for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                  tma_load_2d_pair(b + g * 16384 + j * 8192, &P.mapB, nb + 64 * g, k0 + 64 * j, cbar, keep);
            }
          } else if (P.b_3d) {
            tma_load_3d_pair(b, &P.mapB, 0, nb, k0 / 64, cbar, keep);
          } else {
#pragma unroll
            for (int j = 0; j < kGemmKB; ++j) tma_load_2d_pair(b + j * 16384, &P.mapB, k0 + 64 * j, nb, cbar, keep);
          }
        }
      }
      if (!ok) {
        abort_flag = 1;
        set_error(P.err, DEVERR_TIMEOUT);
        // loads in flight complete on the even CTA's barriers: that CTA
        // drains them (the odd CTA stays resident until then, at the final
        // cluster barrier)
        if (leader)
          for (int k = it - NS < 0 ? 0 : it - NS; k < it; ++k) mbar_wait(full0 + 8 * (k % NS), (k / NS) & 1, drain);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer (the even CTA of a pair) ----
    if (lane == 0 && leader) {
      const uint32_t idesc = idesc_bf16_f32(CL * kGemmM, kGemmN, P.a_mn, P.b_mn);
      // MN-major: atoms of 64 (M or N) x 8 K rows, 64-wide groups 16 KB
      // apart; K-major: atoms of 8 rows x 64 K, K blocks 16 KB apart
      const uint32_t a_lbo = P.a_mn ? 16384 : 16, b_lbo = P.b_mn ? 16384 : 16;
      const uint32_t a_blk = P.a_mn ? 8192 : 16384, b_blk = P.b_mn ? 8192 : 16384;   // next K block
      const uint32_t a_step = P.a_mn ? 2048 : 32, b_step = P.b_mn ? 2048 : 32;         // next 16 of K
      int it = 0, i = 0;
      bool ok = true;
      for (int x = cl; x < nitems && ok; x += ncl, ++i) {
        const GemmItem w = gemm_item(P, x, nslots);
        const int b = i & 1;
        if (i >= 2) {
          // both CTAs' epilogues have drained this accumulator buffer
          bool got = mbar_try_wait_cluster(tempty0 + 8 * b, ((i >> 1) & 1) ^ 1);
          if (!got) {
            const uint64_t t0 = global_ns();
            while (!(got = mbar_try_wait_cluster(tempty0 + 8 * b, ((i >> 1) & 1) ^ 1)))
              if (abort_flag || (int64_t)(global_ns() - t0) > limit) break;
          }
          if (!got) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        const uint32_t d = tmem + b * kGemmN;
        for (int sl = w.sl0; sl < w.sl1; ++sl, ++it) {
          const int s = it % NS;
          if (!gemm_wait(full0 + 8 * s, (it / NS) & 1, limit, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(opnd + s * kStageBytes), bb = a + kHalfA;
#pragma unroll
          for (int j = 0; j < kGemmKB; ++j) {
            const int kb = sl * kGemmKB + j;
            if (kb >= P.nkb) break;
#pragma unroll
            for (int kk = 0; kk < kGemmK / 16; ++kk) {
              const uint64_t ad = smem_desc_sw128(a + j * a_blk + kk * a_step, a_lbo, 1024);
              const uint64_t bd = smem_desc_sw128(bb + j * b_blk + kk * b_step, b_lbo, 1024);
              tc_mma_bf16<CL>(d, ad, bd, idesc, (kb != w.sl0 * kGemmKB) || kk != 0);
            }
          }
          tc_commit<CL>(empty0 + 8 * s);   // both CTAs may refill the slot
        }
        if (!ok) break;
        tc_commit<CL>(tfull0 + 8 * b);
      }
      if (!ok) {
        abort_flag = 1;
        set_error(P.err, DEVERR_TIMEOUT);
      }
      // every MMA issued has completed before either CTA may free TMEM
      tc_commit<CL>(done_bar);
      mbar_wait(done_bar, 0, drain);
    }
  } else if (warp == 2) {
    // ---- epilogue leaf producer ----
    if (lane == 0 && staged && !P.inject) {
      Epi::prefetch(P);
      int g = 0;
      bool ok = true;
      for (int x = cl; x < nitems && ok; x += ncl) {
        int m0, n0;
        tile_of(gemm_item(P, x, nslots).unit, m0, n0);
        for (int j = 0; j < kGemmChunks; ++j, ++g) {
          const int e = g % NE;
          if (g >= NE && !gemm_wait(eempty0 + 8 * e, ((g / NE) & 1) ^ 1, limit, &abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(efull0 + 8 * e, P.epi_tx_bytes);
          Epi::issue(P, smem_u32(ebuf + e * P.epi_stage_bytes), efull0 + 8 * e, m0, n0 + j * kGemmChunk);
        }
      }
      if (!ok) {
        abort_flag = 1;
        set_error(P.err, DEVERR_TIMEOUT);
        for (int k = g - NE < 0 ? 0 : g - NE; k < g; ++k) mbar_wait(efull0 + 8 * (k % NE), (k / NE) & 1, drain);
      }
    }
  } else {
    // ---- epilogue ----
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int rr = q * 32 + lane;        // accumulator row of this thread
    const bool inplace = P.inplace_off >= 0;
    int prev_e = -1;                     // buffer whose release waits for its store (lane 0)

    int g = 0, i = 0;
    bool dead = false;
    for (int x = cl; x < nitems; x += ncl, ++i) {
      const GemmItem w = gemm_item(P, x, nslots);
      int m0, n0;
      tile_of(w.unit, m0, n0);
      const int b = i & 1;
      bool got = gemm_wait(tfull0 + 8 * b, (i >> 1) & 1, limit, &abort_flag);
      tc_fence_after();
      got = __all_sync(0xffffffffu, got);
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + b * kGemmN;
      // a piece: its partial accumulator goes to the workspace; the warp that
      // completes a row block's second piece adds the other and finishes it
      bool finish = true;
      if (w.piece >= 0 && got) {
        // layout [64 column quads][128 rows][4]: a warp's 16-byte accesses
        // cover 512 contiguous bytes
        float4* wq = reinterpret_cast<float4*>(P.ws) + (size_t)(w.q * CL + rank) * (kGemmM * kGemmN / 4) + rr;
#pragma unroll 1
        for (int j = 0; j < kGemmChunks; ++j) {
          float acc[32];
          tmem_ld32(tacc + j * kGemmChunk, acc);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            wq[(size_t)(j * 8 + c) * kGemmM] = make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
        }
        __threadfence();
        __syncwarp();
        int32_t* cnt = P.ws_cnt + ((w.unit - P.nfull) * CL + rank) * 4 + q;
        int last = 0;
        if (lane == 0) last = atomicAdd(cnt, 1) == P.split - 1;
        finish = __shfl_sync(0xffffffffu, last, 0) != 0;
        if (finish) {
          __threadfence();
          if (lane == 0) *cnt = 0;   // every piece has arrived: ready for the next launch
        }
      }
      for (int j = 0; j < kGemmChunks; ++j, ++g) {
        const int e = g % NE;
        if (got && staged) got = gemm_wait(efull0 + 8 * e, (g / NE) & 1, limit, &abort_flag);
        // tcgen05.ld is warp-collective: decide per warp
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          dead = true;
          break;
        }
        if (!finish) {
          // another piece finishes this row block: only release the leaves
          if (lane == 0 && staged) {
            if (inplace) {
              bulk_wait_read<0>();
              if (prev_e >= 0) mbar_arrive(eempty0 + 8 * prev_e);
              prev_e = -1;
            }
            mbar_arrive(eempty0 + 8 * e);
          }
          __syncwarp();
          continue;
        }
        float acc[32], o[32];
        tmem_ld32(tacc + j * kGemmChunk, acc);
        if (w.piece >= 0) {
          // the other piece's partial: two pieces, one addition, the same
          // result whichever finished last
          const float4* oq = reinterpret_cast<const float4*>(P.ws) +
                             (size_t)((w.q ^ 1) * CL + rank) * (kGemmM * kGemmN / 4) + rr;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 t = __ldcg(oq + (size_t)(j * 8 + c) * kGemmM);
            acc[4 * c] = __fadd_rn(acc[4 * c], t.x);
            acc[4 * c + 1] = __fadd_rn(acc[4 * c + 1], t.y);
            acc[4 * c + 2] = __fadd_rn(acc[4 * c + 2], t.z);
            acc[4 * c + 3] = __fadd_rn(acc[4 * c + 3], t.w);
          }
        }
        const uint8_t* st = ebuf + e * P.epi_stage_bytes;
#pragma unroll
        for (int s8 = 0; s8 < 4; ++s8) {
          const GemmEnv env{P, st, rr, m0, n0 + j * kGemmChunk, s8 * 8};
          float a8[8], o8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) a8[k] = acc[s8 * 8 + k];
          Epi::run(env, a8, o8);
#pragma unroll
          for (int k = 0; k < 8; ++k) o[s8 * 8 + k] = o8[k];
        }
        // this warp's 32 rows x 32 columns go out through its own TMA store:
        // no barrier across the epilogue warps
        // the result goes to this warp's rows of the IDENT leaf's chunk (read
        // above, no longer needed) or to a separate double buffer
        uint8_t* ob = inplace ? ebuf + e * P.epi_stage_bytes + P.inplace_off + q * (32 * 128)
                              : obuf + (j & 1) * kGemmOutBytes + q * (32 * 128);
        if (!inplace && lane == 0) bulk_wait_read<1>();   // this buffer's previous store has read it
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4*>(ob + GemmEnv::swz(lane, c)) =
              make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (staged && !inplace) mbar_arrive(eempty0 + 8 * e);
          if (n0 + j * kGemmChunk < P.N && m0 + q * 32 < P.M) {
            tma_store_2d_hint(&P.maps[kMaxStaged], n0 + j * kGemmChunk, m0 + q * 32, smem_u32(ob), l2_evict_first());
          }
          bulk_commit();
          if (inplace) {
            // the previous chunk's buffer is free once its store has read it
            bulk_wait_read<1>();
            if (prev_e >= 0) mbar_arrive(eempty0 + 8 * prev_e);
            prev_e = e;
          }
        }
      }
      if (dead) break;
      // this accumulator buffer may be overwritten by the next tile's MMAs
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(cluster_addr(tempty0 + 8 * b, 0));
      }
    }
    if (dead) {
      abort_flag = 1;
      set_error(P.err, DEVERR_TIMEOUT);
    }
    if (lane == 0) bulk_wait<0>();
  }
  tc_fence_before();
  __syncthreads();
  // no CTA leaves while its peer may still write to its shared memory or
  // issue MMAs into its TMEM
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<CL>(tmem, 512);
}

}  // namespace fg
