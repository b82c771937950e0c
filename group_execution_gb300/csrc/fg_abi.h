// Shared between the host group compiler and the device kernels: the operator
// program format, leaf descriptors and kernel parameter blocks.  Plain data
// only; no std types.
#pragma once
#include <cstdint>
#include <cuda.h>

#ifdef __CUDACC__
#define FG_HD __host__ __device__
#else
#define FG_HD
#endif

namespace fg {

// ---- operator program --------------------------------------------------------
// A group compiles to a postfix program over a small register stack.  The
// host knows the stack depth before every instruction, so each instruction
// carries a dispatch key that already names (operation, depth[, slot]); the
// device switches on it and every register index is a compile-time constant.
constexpr int kMaxDepth = 8;   // stack registers in the largest machine
constexpr int kMaxSlots = 8;   // save slots (values reused inside a group)

enum VmOp : int {
  VM_PUSH_LEAF = 0,  // push leaf `arg` read at this thread's frame points
  VM_PUSH_ACC,       // push the accumulator (GEMM tile value / reduced row value)
  VM_ADD, VM_SUB, VM_MUL, VM_DIV,           // s[d-2] = s[d-2] op s[d-1]; pop
  VM_SCALE, VM_ADDC,                         // s[d-1] = imm*s / s+imm
  VM_RELU, VM_EXP, VM_SIGMOID, VM_TANH, VM_NEG,
  VM_NUM_STACK_OPS,
  // slot ops: PUSH_SLOT pushes slot `arg`; TEE copies the top into slot `arg`;
  // STORE copies the top into slot `arg` and pops.
  VM_PUSH_SLOT = 16, VM_TEE = 17, VM_STORE = 18,
};

// depth before an instruction is 0..kMaxDepth, so keys step by 16
constexpr int kKeyStride = 16;
constexpr int kSlotKeyBase = 256;
FG_HD constexpr int vm_key(int op, int depth) { return op * kKeyStride + depth; }
FG_HD constexpr int vm_slot_key(int op, int slot, int depth) {
  return kSlotKeyBase + (((op - VM_PUSH_SLOT) * kMaxSlots + slot) * kKeyStride + depth);
}

struct VmInstr {
  uint16_t key;   // dispatch key (vm_key / vm_slot_key)
  uint16_t arg;   // leaf index for PUSH_LEAF (slot ops encode the slot in the key)
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

struct LeafDesc {
  int32_t cls;
  int32_t stage_off;     // byte offset of this leaf's boxes inside a stage
  int32_t map_idx;       // tensor map index (staged classes)
  int32_t nterms;        // gather
  const float* ptr;      // gather base pointer (filled at launch)
  int64_t d[kMaxTerms], m[kMaxTerms], s[kMaxTerms];
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
  int32_t* err;                        // device error flag
  int64_t wait_limit_ns;
  int32_t nprog, nepi, nleaves, nstaged;
  int32_t FR, FC;                      // frame
  int32_t ntr, ntc, ntiles;            // tile grid
  int32_t stage_bytes, nstages, tx_bytes;   // stage stride, depth, bytes TMA writes per stage
  int32_t out_tma;                     // 1: output via TMA store, 0: direct stores
  int32_t red_op, nsplit, tiles_per_split, nunits;
};

// GEMM + epilogue kernel.
struct GemmParams {
  CUtensorMap mapA, mapB;              // bf16 operands, MN-major (transA=1 / transB=0)
  CUtensorMap maps[kMaxStaged + 1];    // epilogue leaves, [kMaxStaged] = output
  VmInstr prog[kMaxProg];
  LeafDesc leaves[kMaxLeaves];
  int32_t* err;
  int64_t wait_limit_ns;
  int32_t nprog, nleaves, nstaged;
  int32_t M, N, K;
  int32_t ntm, ntn, ntiles;
  int32_t epi_stage_bytes;
};

// Device error codes written to the flag.
enum DevErr : int { DEVERR_NONE = 0, DEVERR_TIMEOUT = 1, DEVERR_PROGRAM = 2 };

}  // namespace fg
