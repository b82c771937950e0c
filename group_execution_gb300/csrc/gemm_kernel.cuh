// GEMM-epilogue group kernel (K3): D = A * B on the 5th-generation tensor
// cores with the group's elementwise tail applied to the accumulator before
// it ever reaches global memory (TVM "Operator Fusion", Fusion rules, phase
// 0: an out-elementwise-fusable operator such as matmul fuses with its
// elementwise successors; TAG's sufficient-factor gradient G = U^T V is the
// workload).
//
// Persistent: CTAs run in pairs on the SMs of one TPC, and a pair walks
// 256 x TN output tiles (TN = 256, 224 or 128).  Each CTA stages half of
// the tile's A rows and half of its B columns, KB 64-deep K blocks per ring
// slot (two by default: 64 KB), each operand half in one TMA copy where the
// layout allows; the even CTA issues 2-SM tcgen05.mma instructions
// (cta_group::2) that read both CTAs' halves and leave each CTA's 128
// accumulator rows in its own TMEM.  Every operand copy lands in the CTA
// that issued it; no copy is multicast.  Warp roles, in each CTA:
//   warp 0     TMA producer of the bf16 A halves, arming the even CTA's slot
//              barrier; every operand load of both CTAs completes on that
//              barrier,
//   warp 7     TMA producer of the B halves (a slot's copies issue at a few
//              hundred ns each from one thread: two producers halve the time
//              from a slot's release to its refill),
//   warp 1     allocates TMEM (two accumulator buffers, jointly with the
//              peer) and, in the even CTA, issues the MMAs from one thread,
//   warp 2     TMA producer of the epilogue leaves, 128 x 32 chunk by chunk
//              (for long K it also stores the results written in place of an
//              IDENT leaf's chunk, one copy per chunk, before the buffer is
//              loaded again),
//   warps 3-6  epilogue, and warps 8-11 a second set taking the alternate
//              32-column chunks (a chunk's TMEM read, leaf reads and
//              epilogue are one warp's serial chain): each thread owns one
//              accumulator row (TMEM lane), reads 32 columns per chunk with
//              tcgen05.ld, evaluates the epilogue program eight values at a
//              time and stages the result for a TMA store (its own, or, for
//              results written in place with long K, warp 2's).
// The epilogue of tile i overlaps the MMAs of tile i+1.  The last round's
// tiles are cut into column halves (a half-width MMA and B box, over all of
// K, on pairs the round would leave idle), or cut along K: a tile cut along K
// (the last round's, or at a share boundary) meets its two partial
// accumulators in a workspace.  The CTA's last item uses the idle operand
// ring for its stores.  Every wait is bounded; on expiry the CTA records the
// error, drains its copies, frees its TMEM and returns.
#pragma once
#include "fg_device.cuh"

namespace fg {

constexpr int kGemmThreads = kGemmWarps * 32;
constexpr int kGemmABytes = kGemmM * kGemmK * 2;    // 16 KB: this CTA's 128 rows of one A block
constexpr int kGemmOutBytes = kGemmM * kGemmChunk * 4;   // 16 KB

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
    uint32_t f[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = cc0 + q8 + k;
      f[k] = r < P.M && c < P.N ? digit_offset(G, (uint32_t)r * (uint32_t)P.N + (uint32_t)c) : 0u;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = cc0 + q8 + k;
      t[k] = r < P.M && c < P.N ? __ldg(G.ptr + f[k]) : 0.f;
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

// A cluster's work list: item indices [x0, end) in steps of `step`.  Round
// robin: items are whole units, then the pieces of the split last round (two
// K pieces, or the two column halves, of each of its units).
// Stream-K (P.sk): the cluster owns ring slots [b0, b1) of the sequence of
// all units' slots, and its items are the units that range touches.
struct GemmSched {
  int x0, end, step;
  int64_t b0, b1;
};
__device__ __forceinline__ GemmSched gemm_sched(const GemmParams& P, int cl, int ncl, int nslots) {
  GemmSched S;
  if (P.sk) {
    const int64_t W = (int64_t)P.nunits * nslots;
    S.b0 = W * cl / ncl;
    S.b1 = W * (cl + 1) / ncl;
    S.x0 = (int)(S.b0 / nslots);
    S.end = S.b1 > S.b0 ? (int)((S.b1 - 1) / nslots) + 1 : S.x0;
    S.step = 1;
  } else {
    S.b0 = S.b1 = 0;
    S.x0 = cl;
    S.end = P.nfull + (P.nunits - P.nfull) * P.split;
    S.step = ncl;
  }
  return S;
}

// One item: a whole unit, one K piece (ring slots [sl0, sl1)) of a unit cut
// in two, or one column half of a unit (half = 0 or 1, all of K).  q indexes
// a K piece's workspace (q ^ 1 is the other piece of the same unit) and key
// its ready flags.  Of two unequal pieces (a stream-K share boundary, or the
// round-robin tail without ksym) one finishes the unit (fin) and the other
// publishes its partial accumulator; two symmetric pieces both publish and
// each finishes one column half (ehalf).
struct GemmItem {
  int unit, piece, sl0, sl1, q, key;   // piece = -1 for a whole unit or a column half
  int half;                            // -1, or the column half of the unit (a half-width MMA)
  int ehalf;                           // -1, or the column half a symmetric K piece finishes
  bool fin;
};
__device__ __forceinline__ GemmItem gemm_item(const GemmParams& P, const GemmSched& S, int cl, int idx,
                                              int nslots) {
  GemmItem w;
  w.piece = w.q = w.key = w.half = w.ehalf = -1;
  w.fin = true;
  if (P.sk) {
    w.unit = idx;
    const int64_t base = (int64_t)idx * nslots;
    w.sl0 = (int)(S.b0 > base ? S.b0 - base : 0);
    w.sl1 = (int)(S.b1 - base < nslots ? S.b1 - base : nslots);
    if (w.sl0 > 0 || w.sl1 < nslots) {
      // a share boundary cuts this unit: piece 0 ends cluster cl's share
      // (boundary cl + 1), piece 1 starts it (boundary cl)
      w.piece = w.sl0 == 0 ? 0 : 1;
      w.key = (w.piece == 0 ? cl + 1 : cl) - 1;
      w.q = 2 * w.key + w.piece;
      w.fin = w.piece == 0;   // ends the share: its other piece ran first in the next share
    }
  } else if (idx < P.nfull) {
    w.unit = idx;
    w.sl0 = 0;
    w.sl1 = nslots;
  } else if (P.nsplit_n) {
    const int q = idx - P.nfull;
    w.unit = P.nfull + q / 2;
    w.half = q & 1;
    w.sl0 = 0;
    w.sl1 = nslots;
  } else {
    w.q = idx - P.nfull;
    w.unit = P.nfull + w.q / P.split;
    w.key = w.unit - P.nfull;
    w.piece = w.q & 1;
    // symmetric: equal halves of K, each piece finishing one column half;
    // otherwise the first piece is the shorter: it also writes its partial,
    // and is done when the second's MMAs end
    w.sl0 = w.piece ? P.split_at : 0;
    w.sl1 = w.piece ? nslots : P.split_at;
    w.fin = P.ksym || w.piece == 1;
    if (P.ksym) w.ehalf = w.piece;
  }
  return w;
}

// One operand half of a ring slot (this CTA's R rows of A or columns of B,
// KB K blocks from k0) into this CTA's shared memory, counted on the pair
// barrier cbar: one copy through a 3-D view, or 2-D boxes.  Layouts:
// MN-major [R / 64 groups][KB * 64 K rows][64], K-major [KB][R rows][64 K].
template <int KB, int R>
__device__ __forceinline__ void gemm_load_half(uint32_t dst, const CUtensorMap* m, int mn, int v3, int r0, int k0,
                                               uint32_t cbar, uint64_t keep) {
  if (mn) {
    if (v3) {
      tma_load_3d_pair(dst, m, 0, k0, r0 / 64, cbar, keep);
    } else {
#pragma unroll
      for (int g = 0; g < R / 64; ++g)
#pragma unroll
        for (int j = 0; j < KB; ++j)
          tma_load_2d_pair(dst + g * (KB * 8192) + j * 8192, m, r0 + 64 * g, k0 + 64 * j, cbar, keep);
    }
  } else if (v3) {
    tma_load_3d_pair(dst, m, 0, r0, k0 / 64, cbar, keep);
  } else {
#pragma unroll
    for (int j = 0; j < KB; ++j) tma_load_2d_pair(dst + j * (R * 128), m, k0 + 64 * j, r0, cbar, keep);
  }
}

// A CTA pair (a 2-CTA cluster) per 256 x TN tile (cta_group::2), each CTA
// holding half of A's rows and half of B's columns.  KB: K blocks of 64 per
// operand ring slot (1 or 2).  TN: columns of a pair's tile (256; 224, whose
// rounds come out even where 256 leaves a partial last round; or 128:
// half the epilogue per tile, for short K where the epilogue's streams
// dominate and finer tiles fill the last round).
template <class Epi, int KB, int TN>
__device__ __forceinline__ void gemm_body(const GemmParams& P) {
  static_assert(KB == 1 || KB == 2, "one or two K blocks per ring slot");
  static_assert(TN == 256 || TN == 224 || TN == 128, "pair tiles of 256, 224 or 128 columns");
  constexpr int CL = kGemmCluster;                                 // CTAs per cluster: one pair
  constexpr int kBCols = TN / 2;                                   // B columns of the tile per CTA
  // B columns staged per CTA: 224-column tiles stage 128 (whole 64-wide
  // swizzle groups, the ring laid out as for 256) and their MMAs read the
  // first 112
  constexpr int kBStage = TN == 224 ? 128 : kBCols;
  constexpr int kGemmChunks = TN / kGemmChunk;                     // epilogue chunks per tile
  constexpr int kHalfA = KB * kGemmABytes;                         // 128 rows x KB K blocks
  constexpr int kStageBytes = kHalfA + KB * kBStage * kGemmK * 2;  // 32 (24) KB per K block and CTA
  constexpr int kStageBytesH = kHalfA + KB * (kBCols / 2) * kGemmK * 2;   // a column half's slot
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ int issued[2];            // operand slots issued by the A and B producers
  __shared__ uint32_t tmem_slot;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // layout: operand ring | epilogue leaf stages | output staging (per-warp
  // 4 KB boxes, when the result is not written in place) | barriers; the
  // ring and the output staging 1024-byte aligned (128-byte swizzle)
  const int NS = P.nstages, NE = P.n_epi_bufs;
  uint8_t* opnd = smem;
  uint8_t* ebuf = opnd + NS * kStageBytes;
  uint8_t* obuf = ebuf + ((NE * P.epi_stage_bytes + 1023) & ~1023);
  // barriers: full[16] empty[16] tfull[2] tempty[2] efull[8] eempty[8] done
  // last[8] (one per epilogue warp)
  const uint32_t bars = smem_u32(obuf + (P.inplace_off >= 0 ? 0 : 2 * kGemmOutBytes));
  const uint32_t full0 = bars, empty0 = bars + 128, tfull0 = bars + 256, tempty0 = bars + 272;
  const uint32_t efull0 = bars + 288, eempty0 = bars + 352, done_bar = bars + 416, last0 = bars + 424;
  const bool inplace = P.inplace_off >= 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool staged = P.epi_tx_bytes > 0;
  const int nslots = (P.nkb + KB - 1) / KB;                       // ring slots per tile

  const uint32_t rank = cluster_ctarank();
  const int h = (int)(rank & 1);   // CTA within its pair
  const bool leader = h == 0;
  const uint32_t even = 0;         // the pair's MMA-issuing CTA
  // MMA completions arrive at both CTAs of the pair: ring slots are released
  // to both producers, accumulators to both epilogues
  const uint16_t pair_mask = 3u;
  // unit u: the tile of 256 rows in row block u / ntn and TN columns in
  // column block u % ntn; this CTA works on its half h of the rows
  const int ncl = gridDim.x / CL, cl = blockIdx.x / CL;
  const int nsn = P.ntn;
  auto tile_of = [&](int u, int& m0, int& n0) {
    m0 = ((u / nsn) * 2 + h) * kGemmM;
    n0 = (u % nsn) * TN;
  };
  // an item's output block: its unit's tile, or the tile's column half; and
  // its 32-column epilogue chunks
  auto item_tile = [&](const GemmItem& w, int& m0, int& n0) {
    tile_of(w.unit, m0, n0);
    if (w.half > 0) n0 += TN / 2;
  };
  auto item_chunks = [&](const GemmItem& w) { return w.half >= 0 ? kGemmChunks / 2 : kGemmChunks; };
  // the epilogue's view: a symmetric K piece finishes one column half of its
  // (full-width) accumulator
  auto epi_tile = [&](const GemmItem& w, int& m0, int& n0) {
    item_tile(w, m0, n0);
    if (w.ehalf > 0) n0 += TN / 2;
  };
  auto epi_chunks = [&](const GemmItem& w) { return w.ehalf >= 0 ? kGemmChunks / 2 : item_chunks(w); };
  if (threadIdx.x == 0) {
    abort_flag = 0;
    issued[0] = issued[1] = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);   // one commit from the pair's MMA issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 8 * 2);   // every epilogue warp of the pair
    }
    for (int e = 0; e < NE; ++e) {
      mbar_init(efull0 + 8 * e, 1);
      mbar_init(eempty0 + 8 * e, 4);   // the four warps of the chunk's set
    }
    mbar_init(done_bar, 1);
    for (int k = 0; k < 8; ++k) mbar_init(last0 + 8 * k, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc<2>(smem_u32(&tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_launch_dependents();
  pdl_wait();   // the previous grid's writes are visible from here on
  const int64_t limit = P.wait_limit_ns;
  const int64_t drain = limit > kDrainLimitNs ? limit : kDrainLimitNs;
  const GemmSched S = gemm_sched(P, cl, ncl, nslots);

  if (warp == 0 || warp == 7) {
    // ---- operand producers: warp 0 the A halves, warp 7 the B halves ----
    // Ring slot layouts (per CTA), each 128-byte row 128B-swizzled:
    //   K-major operand:  [K block][128 rows][64 K]           (16 KB per K block)
    //   MN-major operand: [64-wide group][KB * 64 K rows][64]  (KB * 8 KB per group)
    const bool isA = warp == 0;
    if (lane == 0 && !P.inject) {
      tma_prefetch(isA ? &P.mapA : &P.mapB);
      if (!isA && P.nsplit_n) tma_prefetch(&P.mapB2);
      const uint64_t keep = l2_evict_last();   // every operand tile is read by several tiles
      // both CTAs' halves are counted on the even CTA's barrier, which the
      // even CTA alone arms with the whole slot's bytes (blocks past K
      // arrive zero-filled and count in full)
      const uint32_t cbar0 = cluster_addr(full0, even), ring = smem_u32(opnd);
      int it = 0, s = 0;
      uint32_t ph = 0;   // ring position and phase parity
      bool ok = true;
      for (int x = S.x0; x < S.end && ok; x += S.step) {
        const GemmItem w = gemm_item(P, S, cl, x, nslots);
        int m0, n0;
        item_tile(w, m0, n0);
        const bool hb = w.half >= 0;   // a column half: each CTA stages kBCols / 2 columns of B
        const int nb = n0 + h * (hb ? kBCols / 2 : kBCols);
        for (int sl = w.sl0; sl < w.sl1; ++sl) {
          if (it >= NS && !gemm_wait(empty0 + 8 * s, ph ^ 1, limit, &abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t a = ring + s * kStageBytes, b = a + kHalfA, cbar = cbar0 + 8 * s, fbar = full0 + 8 * s;
          const int k0 = sl * KB * kGemmK;
          ++it;
          if (++s == NS) {
            s = 0;
            ph ^= 1;
          }
          if (!isA) {
            if constexpr (TN == kGemmN) {
              if (hb) {
                gemm_load_half<KB, kBCols / 2>(b, &P.mapB2, P.b_mn, P.b_3d, nb, k0, cbar, keep);
                continue;
              }
            }
            gemm_load_half<KB, kBStage>(b, &P.mapB, P.b_mn, P.b_3d, nb, k0, cbar, keep);
            continue;
          }
          if (leader) mbar_expect_tx(fbar, 2 * (hb ? kStageBytesH : kStageBytes));
          gemm_load_half<KB, kGemmM>(a, &P.mapA, P.a_mn, P.a_3d, m0, k0, cbar, keep);
        }
      }
      issued[isA ? 0 : 1] = it;
      if (!ok) {
        abort_flag = 1;
        set_error(P.err, DEVERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer (the even CTA of a pair) ----
    if (lane == 0 && leader) {
      const uint32_t idesc = idesc_bf16_f32(2 * kGemmM, TN, P.a_mn, P.b_mn);
      const uint32_t idesc_h = idesc_bf16_f32(2 * kGemmM, TN / 2, P.a_mn, P.b_mn);   // a column half
      // MN-major: atoms of 64 (M or N) x 8 K rows, 64-wide groups 16 KB
      // apart; K-major: atoms of 8 rows x 64 K, K blocks 16 KB apart
      const uint32_t a_lbo = P.a_mn ? KB * 8192 : 16, b_lbo = P.b_mn ? KB * 8192 : 16;
      const uint32_t a_blk = P.a_mn ? 8192 : 16384, b_blk = P.b_mn ? 8192 : kBStage * 128;   // next K block
      const uint32_t b_blk_h = P.b_mn ? 8192 : kBCols / 2 * 128;
      const uint32_t a_step = P.a_mn ? 2048 : 32, b_step = P.b_mn ? 2048 : 32;         // next 16 of K
      // a descriptor's start-address field holds address >> 4 in 14 bits and
      // the ring lies below 2^18 bytes, so descriptors advance by adding
      // offset >> 4: built once here, not per MMA
      const uint32_t ring = smem_u32(opnd);
      const uint64_t ad0 = smem_desc_sw128(ring, a_lbo, 1024), bd0 = smem_desc_sw128(ring + kHalfA, b_lbo, 1024);
      uint32_t aoff[KB * 4], boff[KB * 4], boff_h[KB * 4];
#pragma unroll
      for (int j = 0; j < KB; ++j)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          aoff[j * 4 + kk] = (j * a_blk + kk * a_step) >> 4;
          boff[j * 4 + kk] = (j * b_blk + kk * b_step) >> 4;
          boff_h[j * 4 + kk] = (j * b_blk_h + kk * b_step) >> 4;
        }
      int s = 0, i = 0;
      uint32_t ph = 0;   // ring position and phase parity
      bool ok = true;
      for (int x = S.x0; x < S.end && ok; x += S.step, ++i) {
        const GemmItem w = gemm_item(P, S, cl, x, nslots);
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
        const uint32_t d = tmem + b * TN;
        const bool hb = w.half >= 0;
        const uint32_t id = hb ? idesc_h : idesc;
        for (int sl = w.sl0; sl < w.sl1; ++sl) {
          if (!gemm_wait(full0 + 8 * s, ph, limit, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t so = (uint32_t)(s * kStageBytes) >> 4;
          const int nk = P.nkb - sl * KB;   // K blocks left (the last slot may hold fewer than KB)
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            if (j >= nk) break;
#pragma unroll
            for (int kk = 0; kk < kGemmK / 16; ++kk)
              tc_mma_bf16<2>(d, ad0 + so + aoff[j * 4 + kk], bd0 + so + (hb ? boff_h : boff)[j * 4 + kk], id,
                             sl != w.sl0 || j != 0 || kk != 0);
          }
          tc_commit_mask(empty0 + 8 * s, pair_mask);   // both producers may refill the slot
          if (++s == NS) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_mask(tfull0 + 8 * b, pair_mask);
      }
      if (!ok) {
        abort_flag = 1;
        set_error(P.err, DEVERR_TIMEOUT);
      }
      // every MMA issued has completed before either CTA may free TMEM
      tc_commit_mask(done_bar, pair_mask);
      mbar_wait(done_bar, 0, drain);
    }
  } else if (warp == 2) {
    // ---- epilogue leaf producer ----
    if (lane == 0 && staged && !P.inject) {
      Epi::prefetch(P);
      // the oldest chunk whose buffer has not been taken back: item rx,
      // column chunk rj; its results leave from the buffer (in place) when
      // this CTA finishes the unit and it is not the CTA's last item (whose
      // results go out from the operand ring, warp by warp)
      const bool pstore = inplace && !P.wstore;   // this thread stores in-place results
      int rx = S.x0, rj = 0, rm0 = 0, rn0 = 0, rnch = kGemmChunks;
      bool rstore = false;
      auto retire_item = [&]() {
        if (rx >= S.end) return;
        const GemmItem w = gemm_item(P, S, cl, rx, nslots);
        epi_tile(w, rm0, rn0);
        rnch = epi_chunks(w);
        rstore = (w.piece < 0 || w.fin) && (rx + S.step < S.end || !P.last_ring);
      };
      // wait until chunk h's buffer is released by its four epilogue warps,
      // store the results they left in it, and move on to the next chunk
      auto retire = [&](int h) -> bool {
        const int e = h % NE;
        if (!gemm_wait(eempty0 + 8 * e, (h / NE) & 1, limit, &abort_flag)) return false;
        if (rstore && rn0 + rj * kGemmChunk < P.N && rm0 < P.M) {
          tma_store_2d_hint(&P.maps[kMaxStaged + 1], rn0 + rj * kGemmChunk, rm0,
                            smem_u32(ebuf + e * P.epi_stage_bytes + P.inplace_off), l2_evict_first());
          bulk_commit();
        }
        if (++rj == rnch) {
          rj = 0;
          rx += S.step;
          retire_item();
        }
        return true;
      };
      if (pstore) retire_item();
      int g = 0;
      bool ok = true;
      for (int x = S.x0; x < S.end && ok; x += S.step) {
        const GemmItem wi = gemm_item(P, S, cl, x, nslots);
        int m0, n0;
        epi_tile(wi, m0, n0);
        const int nch = epi_chunks(wi);
        for (int j = 0; j < nch; ++j, ++g) {
          const int e = g % NE;
          if (g >= NE) {
            if (pstore ? !retire(g - NE)
                       : !gemm_wait(eempty0 + 8 * e, ((g / NE) & 1) ^ 1, limit, &abort_flag)) {
              ok = false;
              break;
            }
            if (pstore) bulk_wait_read<0>();   // a store from this buffer has read it
          }
          mbar_expect_tx(efull0 + 8 * e, P.epi_tx_bytes);
          Epi::issue(P, smem_u32(ebuf + e * P.epi_stage_bytes), efull0 + 8 * e, m0, n0 + j * kGemmChunk);
        }
      }
      // the last chunks' results (only in place: otherwise nothing waits for
      // these releases)
      for (int h = g - NE < 0 ? 0 : g - NE; ok && pstore && h < g; ++h) ok = retire(h);
      if (!ok) {
        abort_flag = 1;
        set_error(P.err, DEVERR_TIMEOUT);
        for (int k = g - NE < 0 ? 0 : g - NE; k < g; ++k) mbar_wait(efull0 + 8 * (k % NE), (k / NE) & 1, drain);
      }
      bulk_wait<0>();   // the stores issued here have completed
    }
  } else {
    // ---- epilogue ----
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int set = warp >= 8 ? 1 : 0;   // chunks j with j % 2 == set
    const int ew = set * 4 + q;          // epilogue warp index
    const int rr = q * 32 + lane;        // accumulator row of this thread
    // in place with per-warp stores: a chunk's buffer is released once this
    // warp's copy has read it, checked at the warp's next store
    const bool wdefer = inplace && P.wstore;
    int prev_e = -1;                     // buffer whose release waits for its store (lane 0)

    int g = 0, i = 0;
    bool dead = false;
    for (int x = S.x0; x < S.end; x += S.step, ++i) {
      const GemmItem w = gemm_item(P, S, cl, x, nslots);
      int m0, n0;
      epi_tile(w, m0, n0);
      const int nch = epi_chunks(w);
      const int tc0 = w.ehalf >= 0 ? w.ehalf * (kGemmChunks / 2) : 0;   // first accumulator chunk of this view
      const int b = i & 1;
      bool got = gemm_wait(tfull0 + 8 * b, (i >> 1) & 1, limit, &abort_flag);
      tc_fence_after();
      got = __all_sync(0xffffffffu, got);
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + b * TN;
      // a piece of a unit cut in two: the piece that runs first puts its
      // partial accumulator (this warp's 32 rows) in the workspace and raises
      // the rows' ready flag; the other waits for the flag, adds the partial
      // and runs the epilogue
      bool finish = true;
      if (w.ehalf >= 0 && got) {
        // a symmetric K piece: this piece's partial of the other column half
        // into the workspace ([32 column quads][128 rows][4]: a warp's
        // 16-byte stores cover 512 contiguous bytes), this warp's flag
        // raised, then the other piece's partial of this half awaited
        // (bounded: it runs on another cluster)
        float4* wq = reinterpret_cast<float4*>(P.ws) + (size_t)(w.q * CL + rank) * (kGemmM * TN / 4) + rr;
        const int oc0 = (1 - w.ehalf) * (kGemmChunks / 2);
#pragma unroll 1
        for (int j = set; j < kGemmChunks / 2; j += 2) {
          float acc[32];
          tmem_ld32(tacc + (oc0 + j) * kGemmChunk, acc);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            wq[(size_t)(j * 8 + c) * kGemmM] = make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
        }
        __threadfence();
        __syncwarp();
        int32_t* mine = P.ws_cnt + ((w.key * 2 + w.piece) * CL + rank) * 8 + ew;
        int32_t* other = P.ws_cnt + ((w.key * 2 + (1 - w.piece)) * CL + rank) * 8 + ew;
        int ready = 0;
        if (lane == 0) {
          st_release_gpu(mine, 1);
          const uint64_t t0 = global_ns();
          while (!(ready = ld_acquire_gpu(other) == 1))
            if (abort_flag || (int64_t)(global_ns() - t0) > limit) break;
          if (ready) *other = 0;   // consumed: clear for the next launch
        }
        got = __shfl_sync(0xffffffffu, ready, 0) != 0;
        __syncwarp();   // orders the other lanes' partial loads after lane 0's acquire
      } else if (w.piece >= 0 && got) {
        int32_t* flag = P.ws_cnt + (w.key * CL + rank) * 8 + ew;
        if (!w.fin) {
          // layout [64 column quads][128 rows][4]: a warp's 16-byte accesses
          // cover 512 contiguous bytes
          float4* wq = reinterpret_cast<float4*>(P.ws) + (size_t)(w.q * CL + rank) * (kGemmM * TN / 4) + rr;
#pragma unroll 1
          for (int j = set; j < kGemmChunks; j += 2) {
            float acc[32];
            tmem_ld32(tacc + j * kGemmChunk, acc);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              wq[(size_t)(j * 8 + c) * kGemmM] = make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) st_release_gpu(flag, 1);
          finish = false;
        } else {
          // the other piece runs on another cluster and never waits for this
          // one: a bounded wait
          int ready = 0;
          if (lane == 0) {
            const uint64_t t0 = global_ns();
            while (!(ready = ld_acquire_gpu(flag) == 1))
              if (abort_flag || (int64_t)(global_ns() - t0) > limit) break;
            if (ready) *flag = 0;   // consumed: clear for the next launch
          }
          got = __shfl_sync(0xffffffffu, ready, 0) != 0;
          __syncwarp();   // orders the other lanes' partial loads after lane 0's acquire
        }
      }
      // The CTA's last item: every MMA has completed, so the operand ring is
      // idle; each TMEM lane quarter takes TN * 128 bytes of it (when the
      // ring is at least four times that) for the other piece's partial and
      // the result chunks, so that no chunk waits for a store buffer.
      const bool last = P.last_ring && x + S.step >= S.end;
      uint8_t* wring = opnd + q * (TN * 128);
      if (last && wdefer && lane == 0 && prev_e >= 0) {
        bulk_wait_read<0>();
        mbar_arrive(eempty0 + 8 * prev_e);
        prev_e = -1;
      }
      const float4* oq = nullptr;   // the other piece's partial (finishing a piece)
      bool part_smem = false;
      float4 nxt[8];
      if (w.piece >= 0 && finish && got) {
        oq = reinterpret_cast<const float4*>(P.ws) + (size_t)((w.q ^ 1) * CL + rank) * (kGemmM * TN / 4) + rr;
        if (last && w.ehalf < 0) {
          // this warp's rows of the partial in its chunks, [column quad][32
          // rows][16 B]: one 512-byte bulk copy per lane and column quad
          const uint32_t lbar = last0 + 8 * ew;
          if (lane == 0) mbar_expect_tx(lbar, TN / 8 * 512);
          __syncwarp();
          if (lane < TN / 8) {
            const int c = ((lane >> 3) * 2 + set) * 8 + (lane & 7);
            bulk_load(smem_u32(wring) + c * 512, oq - lane + (size_t)c * kGemmM, 512, lbar);
          }
          got = __all_sync(0xffffffffu, gemm_wait(lbar, 0, limit, &abort_flag));
          part_smem = true;
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) nxt[c] = __ldcg(oq + (size_t)(set * 8 + c) * kGemmM);
        }
      }
      const bool inpl = inplace && !last;   // results in place in the leaf chunk
      for (int j = 0; j < nch; ++j, ++g) {
        if ((j & 1) != set) continue;   // the other set's chunk
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
            if (inpl && wdefer && prev_e >= 0) {
              bulk_wait_read<0>();
              mbar_arrive(eempty0 + 8 * prev_e);
              prev_e = -1;
            }
            mbar_arrive(eempty0 + 8 * e);
          }
          __syncwarp();
          continue;
        }
        float acc[32], o[32];
        tmem_ld32(tacc + (tc0 + j) * kGemmChunk, acc);
        if (oq) {
          // the other piece's partial: two pieces, one addition, the same
          // result whichever finished last; from the ring, or with the next
          // chunk's loads issued before this chunk is used (each is an L2
          // round trip)
          float4 cur[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            cur[c] = part_smem ? *reinterpret_cast<const float4*>(wring + (j * 8 + c) * 512 + lane * 16) : nxt[c];
          if (!part_smem && j + 2 < nch) {
#pragma unroll
            for (int c = 0; c < 8; ++c) nxt[c] = __ldcg(oq + (size_t)((j + 2) * 8 + c) * kGemmM);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            acc[4 * c] = __fadd_rn(acc[4 * c], cur[c].x);
            acc[4 * c + 1] = __fadd_rn(acc[4 * c + 1], cur[c].y);
            acc[4 * c + 2] = __fadd_rn(acc[4 * c + 2], cur[c].z);
            acc[4 * c + 3] = __fadd_rn(acc[4 * c + 3], cur[c].w);
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
        // the result goes to this warp's rows of the IDENT leaf's chunk (read
        // above, no longer needed), to a separate buffer or, in the last
        // item, to the chunk's 4 KB of the ring (whose partial has been read:
        // all lanes read before any writes, below); it leaves through this
        // warp's own TMA store of its 32 rows x 32 columns, or (in place,
        // long K) through warp 2's store of the whole chunk
        uint8_t* ob = last   ? wring + j * 4096
                      : inpl ? ebuf + e * P.epi_stage_bytes + P.inplace_off + q * (32 * 128)
                             : obuf + (j & 1) * kGemmOutBytes + q * (32 * 128);
        if (!inpl && !last && lane == 0) bulk_wait_read<0>();   // this warp's buffer: its previous store has read it
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4*>(ob + GemmEnv::swz(lane, c)) =
              make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (staged && !inpl) mbar_arrive(eempty0 + 8 * e);   // the leaf chunk has been read
          if (!inpl || P.wstore) {
            if (n0 + j * kGemmChunk < P.N && m0 + q * 32 < P.M) {
              tma_store_2d_hint(&P.maps[kMaxStaged], n0 + j * kGemmChunk, m0 + q * 32, smem_u32(ob), l2_evict_first());
            }
            bulk_commit();
          }
          if (inpl && !wdefer) {
            mbar_arrive(eempty0 + 8 * e);   // warp 2 stores the chunk before reloading the buffer
          } else if (inpl && NE > 2) {
            // this warp's previous chunk's buffer is free once its copy has
            // read it (a wait here would stall the warp for every copy)
            bulk_wait_read<1>();
            if (prev_e >= 0) mbar_arrive(eempty0 + 8 * prev_e);
            prev_e = e;
          } else if (inpl) {
            // with two leaf buffers each set's chunks reuse one buffer: free
            // it now (a deferred release would wait for itself)
            bulk_wait_read<0>();
            mbar_arrive(eempty0 + 8 * e);
          }
        }
      }
      if (dead) break;
      // this accumulator buffer may be overwritten by the next tile's MMAs
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(cluster_addr(tempty0 + 8 * b, even));
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
  if (abort_flag && leader && threadIdx.x == 0) {
    // loads in flight complete on the even CTA's barriers: that CTA drains
    // the slots either producer may still be filling (the odd CTA stays
    // resident until then, at the cluster barrier below)
    const int last = issued[0] > issued[1] ? issued[0] : issued[1];
    for (int k = last - NS < 0 ? 0 : last - NS; k < last; ++k) mbar_wait(full0 + 8 * (k % NS), (k / NS) & 1, drain);
  }
  // no CTA leaves while its peer may still write to its shared memory or
  // issue MMAs into its TMEM
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<2>(tmem, 512);
}

}  // namespace fg
