// Shared between the host group compiler and the device kernels: the operator
// program format, leaf descriptors and kernel parameter blocks.  Plain data
// only; no std types.
#pragma once
#ifdef __CUDACC_RTC__
// compiled at run time by NVRTC: no system headers
typedef unsigned char uint8_t;
typedef unsigned short uint16_t;
typedef unsigned int uint32_t;
typedef unsigned long long uint64_t;
typedef int int32_t;
typedef long long int64_t;
typedef unsigned long long uintptr_t;
struct alignas(128) CUtensorMap {
  unsigned long long opaque[16];
};
#else
#include <cstdint>
#include <cuda.h>
#endif

#ifdef __CUDACC__
#define FG_HD __host__ __device__
#else
#define FG_HD
#endif

namespace fg {

// ---- operator program --------------------------------------------------------
// A group compiles to a postfix program over a small register stack.  The
// host knows the stack depth before every instruction, so each instruction
// carries a dense case number that already names (operation, depth[, slot]);
// the device switches on it and every register index is a compile-time
// constant.  Binary operators also come in forms whose right operand is a
// leaf or a save slot, which saves a push.
constexpr int kMaxDepth = 8;   // stack registers in the largest machine
constexpr int kMaxSlots = 8;   // save slots (values reused inside a group)

enum VmOp : int {
  VM_PUSH_LEAF = 0,  // push leaf `arg` read at this thread's frame points
  VM_PUSH_ACC,       // push the accumulator (GEMM tile value / reduced row value)
  VM_ADD, VM_SUB, VM_MUL, VM_DIV,           // TOP = below op TOP; pop
  VM_SCALE, VM_ADDC,                         // TOP = imm*TOP / TOP+imm
  VM_RELU, VM_EXP, VM_SIGMOID, VM_TANH, VM_NEG,
  VM_ADD_L, VM_SUB_L, VM_MUL_L, VM_DIV_L,    // TOP = TOP op leaf[arg]
  VM_ADD_S, VM_SUB_S, VM_MUL_S, VM_DIV_S,    // TOP = TOP op slot
  VM_PUSH_SLOT,      // push slot
  VM_TEE,            // copy TOP into slot
  VM_STORE,          // copy TOP into slot and pop
};

// Dense case numbers (no holes, so the device switch is one jump table).
constexpr int kCaseLeaf = 0;                                // + d, d in [0, 8)
constexpr int kCaseAcc = kCaseLeaf + kMaxDepth;             // + d
constexpr int kCaseBin = kCaseAcc + kMaxDepth;              // + (op-ADD)*(8-1) + (d-2), d in [2, 8]
constexpr int kCaseUn = kCaseBin + 4 * (kMaxDepth - 1);     // + (op-SCALE)
constexpr int kCaseBinL = kCaseUn + 7;                      // + (op-ADD_L)
constexpr int kCaseBinS = kCaseBinL + 4;                    // + (op-ADD_S)*8 + s
constexpr int kCasePushS = kCaseBinS + 4 * kMaxSlots;       // + s*8 + d, d in [0, 8)
constexpr int kCaseTee = kCasePushS + kMaxSlots * kMaxDepth;  // + s
constexpr int kCaseStore = kCaseTee + kMaxSlots;            // + s*8 + (d-1), d in [1, 8]
constexpr int kNumCases = kCaseStore + kMaxSlots * kMaxDepth;

FG_HD constexpr int vm_case(int op, int depth, int slot) {
  return op == VM_PUSH_LEAF ? kCaseLeaf + depth
       : op == VM_PUSH_ACC ? kCaseAcc + depth
       : op <= VM_DIV ? kCaseBin + (op - VM_ADD) * (kMaxDepth - 1) + (depth - 2)
       : op <= VM_NEG ? kCaseUn + (op - VM_SCALE)
       : op <= VM_DIV_L ? kCaseBinL + (op - VM_ADD_L)
       : op <= VM_DIV_S ? kCaseBinS + (op - VM_ADD_S) * kMaxSlots + slot
       : op == VM_PUSH_SLOT ? kCasePushS + slot * kMaxDepth + depth
       : op == VM_TEE ? kCaseTee + slot
       : kCaseStore + slot * kMaxDepth + (depth - 1);
}

struct VmInstr {
  uint16_t key;   // dense case number (vm_case)
  uint16_t arg;   // leaf index for PUSH_LEAF and the *_L forms
  float imm;      // SCALE / ADDC immediate
};

// ---- leaves ------------------------------------------------------------------
// Where a leaf value is read for frame point (r, c).  Maps are digit forms
// over the frame's flat index g = r*FC + c:  f = sum_k ((g / d_k) % m_k) * s_k.
// Four of them are staged through shared memory by TMA:
enum LeafClass : int {
  LEAF_IDENT = 0,   // f = g           (same row-major order as the frame)
  LEAF_TRANS = 1,   // f = c*FR + r    (leaf is the frame transposed)
  LEAF_COL = 2,     // f = c           (vector indexed by frame column)
  LEAF_ROW = 3,     // f = r           (vector indexed by frame row)
  LEAF_GATHER = 4,  // anything else: per-element loads from global memory
};

constexpr int kMaxTerms = 4;

// Division by an invariant divisor d of dividends x < 2^31 (Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication"):
// floor(x / d) = floor(x * mul / 2^sh) with l = ceil(log2 d),
// mul = ceil(2^(31 + l) / d) < 2^32 and sh = 31 + l.  With x < 2^31,
// x * mul / 2^sh exceeds x / d by less than 2^-l <= 1/d, which never
// reaches the next integer.  A divisor above 2^31 gives mul = 0 (quotient 0).
struct FastDiv {
  uint32_t mul;
  int32_t sh;
};
#ifndef __CUDACC_RTC__
inline FastDiv fast_div(int64_t d) {
  FastDiv f{0u, 32};
  if (d <= 0 || d > (int64_t(1) << 31)) return f;
  int l = 0;
  while ((int64_t(1) << l) < d) ++l;
  const uint64_t num = uint64_t(1) << (31 + l);
  f.mul = (uint32_t)((num + (uint64_t)d - 1) / (uint64_t)d);
  f.sh = 31 + l;
  return f;
}
#endif

struct LeafDesc {
  int32_t cls;
  int32_t stage_off;     // byte offset of this leaf's boxes inside a stage
  int32_t map_idx;       // tensor map index (staged classes)
  int32_t nterms;        // gather
  const float* ptr;      // gather base pointer (filled at launch)
  int64_t d[kMaxTerms], m[kMaxTerms], s[kMaxTerms];
  FastDiv dd[kMaxTerms], dm[kMaxTerms];   // the divisions by d[k] and m[k]
  // a tuple's field is read at g - shift (staged boxes move by shift_r rows
  // and shift_c columns); gathers skip indices outside [0, numel)
  int64_t shift, numel;
  int32_t shift_r, shift_c;
};

// An extra output of a multi-output group (a value computed inside the group
// that is also needed outside it): written at frame point g to
// f = sum_k ((g / d_k) % m_k) * s_k, a permutation of its elements; cls is
// LEAF_IDENT (f = g), LEAF_TRANS (f = c*FR + r) or LEAF_GATHER (the digits).
constexpr int kMaxXOut = 4;
struct XOutDesc {
  float* ptr;            // filled at launch
  int32_t cls, nterms;
  int64_t d[kMaxTerms], m[kMaxTerms], s[kMaxTerms];
  FastDiv dd[kMaxTerms], dm[kMaxTerms];
};

// ---- kernel parameter blocks -------------------------------------------------
constexpr int kMaxStaged = 16;    // TMA-staged leaves per group
constexpr int kMaxLeaves = 24;    // all leaf reads (staged + gathered)
constexpr int kMaxProg = 448;     // instructions in the main program
constexpr int kMaxEpi = 64;       // instructions in a reduce epilogue
constexpr int kMaxEpiLeaves = 8;

// Elementwise / reduce group kernels (tile = 32 frame rows x 64 frame cols).
constexpr int kTileR = 32;
constexpr int kTileC = 64;
constexpr int kConsumerWarps = 8;
constexpr int kProducerWarps = 2;     // group kernels: TMA producers taking alternate tiles
constexpr int kMaxStages = 16;
constexpr int kSmallThreads = 128;     // direct kernel: four warps, one frame row segment each
constexpr int64_t kSmallGroupBytes = 2 << 20;   // groups of at most this many algorithmic bytes run it
constexpr int kDirectMinWarps = 8192;  // larger row reductions run it from this many row segments

enum RedOp : int { RED_NONE = 0, RED_SUM = 1, RED_MAX = 2 };

struct GroupParams {
  CUtensorMap maps[kMaxStaged + 1];    // staged leaves, then [kMaxStaged] = output
  VmInstr prog[kMaxProg];
  LeafDesc leaves[kMaxLeaves];
  VmInstr epi[kMaxEpi];                // reduce epilogue (on the reduced vector)
  const float* epi_leaf[kMaxEpiLeaves];
  float* out;                          // output base (direct stores / reduce output)
  float* scratch;                      // reduce split partials [nsplit][FR]
  int32_t* counters;                   // reduce split arrival counters [ntr]
  unsigned long long* sched;           // elementwise groups: tiles claimed by all launches (claim c: tile
                                       // first + c mod ntiles)
  int32_t* err;                        // device error flag
  int64_t wait_limit_ns;
  int32_t nprog, nepi, nleaves, nstaged;
  int32_t FR, FC;                      // frame
  int32_t ntr, ntc, ntiles;            // tile grid
  int32_t stage_bytes, nstages, tx_bytes;   // stage stride, depth, bytes TMA writes per stage
  int32_t out_tma;                     // 1: CTA tile via smem + TMA store, 2: per-warp TMA slices, 0: direct stores
  int32_t band;                        // tile order: 0 row-major, else bands of `band` tile rows
  int32_t red_op, nsplit, tiles_per_split, nunits;
  int32_t inject;                      // failure injection: 1 = the producer issues no loads
  int32_t nxout;                       // extra outputs (compiled programs only)
  int32_t xout_tma;                    // 1: each warp stages its slice of every extra output
                                       //    in shared memory and stores it with TMA (xmaps)
  int32_t seg, seg_cols;               // direct kernel: warps per frame row (1, 2 or 4), columns per
                                       //    warp's segment (a multiple of 256 unless one segment)
  XOutDesc xout[kMaxXOut];
  CUtensorMap xmaps[kMaxXOut];
};

// GEMM + epilogue kernel: 128 x 256 accumulator tiles in TMEM, K in blocks
// of 64, the epilogue in 128 x 32 column chunks.
constexpr int kGemmM = 128, kGemmN = 256, kGemmK = 64, kGemmChunk = 32;
constexpr int kGemmKB = 2;             // K blocks per operand ring slot (interpreted kernel; compiled: 1 or 2)
constexpr int kGemmWarps = 12;         // A loads, MMA, epilogue loads, 4 epilogue warps, B loads, 4 epilogue warps
constexpr int kGemmCluster = 2;        // CTAs of a pair issuing 2-SM MMAs on one 256-row tile

struct GemmParams {
  CUtensorMap mapA, mapB;              // bf16 operands (boxes per major-ness)
  CUtensorMap mapB2;                   // B in half-width boxes (units cut into column halves)
  CUtensorMap maps[kMaxStaged + 2];    // epilogue leaves, [kMaxStaged] = output in 32 x 32 boxes,
                                       // [kMaxStaged + 1] = output in 128 x 32 boxes
  VmInstr prog[kMaxProg];              // epilogue program (interpreted variant)
  LeafDesc leaves[kMaxLeaves];
  float* out;
  int32_t* err;
  int64_t wait_limit_ns;
  int32_t nprog, nleaves, nstaged;
  int32_t M, N, K;
  int32_t ntm, ntn, ntiles, nkb;
  int32_t a_mn, b_mn;                  // 1: operand stored MN-major (M or N contiguous)
  int32_t a_3d, b_3d;                  // 1: the operand's half tile of a ring slot comes in one
                                       //    copy through a 3-D map (MN-major: [groups][K][64],
                                       //    K-major: [K blocks][rows][64])
  int32_t nstages;                     // operand ring depth
  int32_t epi_stage_bytes, epi_tx_bytes, n_epi_bufs;
  int32_t inplace_off;                 // >= 0: the result overwrites this IDENT leaf's chunk (no out buffers)
  int32_t wstore;                      // in place: 1 = each epilogue warp stores its rows of the chunk and
                                       // frees the buffer once the copy has read them (checked at its next
                                       // store); 0 = the leaf producer stores the whole chunk before
                                       // reloading the buffer
  int32_t inject;                      // failure injection: 1 = the producers issue no loads
  int32_t last_ring;                   // 1: the CTA's last item stages its results in the idle operand
                                       // ring (which holds 4 x TN x 128 bytes); 0: as every other item
  // work units: the pairs' 256-row x TN-column tiles in row-major order
  int32_t nunits;
  // round-robin schedule: units [0, nfull) run whole; each later unit runs
  // as split = 2 pieces along K, ring slots [0, split_at) and
  // [split_at, nslots); without ksym the first publishes its partial
  // accumulator in the workspace and the second adds it and runs the
  // epilogue
  int32_t nfull, split, split_at;
  // nsplit_n = 1: the split units are cut into their two column halves
  // instead (each over all of K, on a pair of its own: no partial sums)
  int32_t nsplit_n;
  // sk = 1: each cluster runs a contiguous 1/ncl share of all units' ring
  // slots instead (at least one whole unit, so a unit is cut at most once,
  // into the two pieces on either side of a share boundary)
  int32_t sk;
  // ksym = 1 (round robin with K pieces): the two pieces of a cut unit take
  // equal halves of K and each finishes one column half of the tile: each
  // writes its partial of the other's half, raises its flags, then waits for
  // the other's partial of its own half (neither waits before publishing)
  int32_t ksym;
  float* ws;                           // [pieces][cluster CTAs][64 column quads][128 rows][4] partial accumulators
  int32_t* ws_cnt;                     // [split units][pieces (ksym)][cluster CTAs][8 epilogue warps]
                                       // partial-ready flags (cleared by the reader)
};

// Loads already issued always land; waiting for them before a CTA exits uses
// at least this bound, whatever the user's wait limit.
constexpr int64_t kDrainLimitNs = 100000000LL;

// Device error codes written to the flag.
enum DevErr : int { DEVERR_NONE = 0, DEVERR_TIMEOUT = 1, DEVERR_PROGRAM = 2 };

}  // namespace fg
