// Host-side graph IR, grouping and group compilation (internal header).
#pragma once
#include <cstdint>
#include <functional>
#include <string>
#include <vector>

#include "groupexec.h"
#include "fg_abi.h"

namespace fg {

enum Kind : int32_t {
  K_ELEMWISE = 0, K_BROADCAST = 1, K_INJECTIVE = 2, K_COMM_REDUCE = 3,
  K_OUT_EWISE_FUSABLE = 4, K_TUPLE = 7, K_OPAQUE = 8
};

// The pattern kind of every operator (TVM "Operator Fusion", Operator Pattern
// Classification: bias_add is broadcast, transpose/reshape injective, sum/max
// commutative reduce, matmul out-elementwise-fusable, side effects opaque).
Kind op_kind(int op);

struct Value {
  int32_t dtype = FG_F32;
  int32_t ndim = 2;
  int64_t rows = 1, cols = 1;   // rank-1 values: rows = 1, cols = n
  bool is_input = true;
  int32_t node = -1;            // producing node, -1 for graph inputs
  int64_t numel() const { return rows * cols; }
  int64_t bytes() const { return numel() * (dtype == FG_BF16 ? 2 : 4); }
  bool same_shape(const Value& o) const { return ndim == o.ndim && rows == o.rows && cols == o.cols; }
};

struct Node {
  int32_t op = 0;
  std::vector<int32_t> args;    // value ids
  std::vector<float> attrs;
  int32_t value = -1;           // output value id
};

struct Graph {
  std::vector<Value> values;
  std::vector<Node> nodes;
  std::vector<char> is_output;  // per value
};

// Maps: f = sum_k ((g / d_k) % m_k) * s_k over the frame flat index g, with
// the terms tiling the value's index range (s_0 = 1, s_{k+1} = s_k * m_k).
// A map may also carry a shift: it is evaluated at g - shift (a field of a
// tuple read at the tuple's frame point).
struct Map {
  int n = 0;
  int64_t d[kMaxTerms] = {0}, m[kMaxTerms] = {0}, s[kMaxTerms] = {0};
  int64_t shift = 0;
  bool operator==(const Map& o) const;
};

struct LeafUse {            // one (value, map) read by a program
  int32_t value;
  Map map;
  int32_t cls;              // LeafClass
  int64_t numel;            // elements of the value (bounds of shifted gathers)
};

// One node of a group's expression DAG (children before parents).
struct JExpr {
  int kind;          // 0 leaf, 1 accumulator, 2 unary, 3 binary, 4 select
  int vm;            // VmOp of the operation (select: 0 = by frame row, 1 = by frame column)
  float imm;
  int a, b;          // children (select: a where the row / column is below `leaf`, else b)
  int leaf;          // leaf index (kind 0), bound (kind 4)
};

struct CompiledGroup {
  int32_t exec = FG_EXEC_ELEMWISE;   // fg_exec_kind
  std::vector<int32_t> nodes;         // ascending node ids
  int32_t sink = -1;                  // sink node
  int32_t out_value = -1;
  // extra outputs (values of the group also read outside it): value, map
  // from the frame, and the expression that computes it
  std::vector<int32_t> xout_values;
  std::vector<Map> xout_maps;
  std::vector<int> xout_cls;          // LEAF_IDENT, LEAF_TRANS or LEAF_GATHER (any other permutation)
  int xout_tma = 0;                   // extra outputs staged per warp and stored by TMA (plan_staging)
  std::vector<int> xout_expr;
  std::vector<int32_t> leaf_values;   // distinct outside values, first-use order
  int64_t alg_bytes = 0, alg_flops = 0;
  int64_t FR = 1, FC = 1;             // frame
  // main program (K1: whole group; K2: prologue; K3: epilogue)
  std::vector<VmInstr> prog;
  std::vector<LeafUse> leaves;
  std::vector<JExpr> dag;             // expression DAG of the main program
  int dag_root = -1;
  std::vector<JExpr> epi_dag;         // reduce epilogue DAG (leaves index epi_leaf_values)
  int epi_root = -1;
  int depth = 0, slots = 0;
  bool needs_jit = false;             // selects (tuples): no interpreter program
  // reduce
  int32_t red_op = RED_NONE;
  std::vector<VmInstr> epi;
  std::vector<int32_t> epi_leaf_values;
  int epi_depth = 0, epi_slots = 0;
  // gemm
  int32_t mm_a = -1, mm_b = -1, mm_ta = 0, mm_tb = 0;
  int64_t M = 0, N = 0, K = 0;
  int gemm_kb = 2;                    // K blocks of 64 per operand ring slot
  int gemm_tn = 256;                  // columns of a pair's tile
  // staging decisions (filled by plan_staging)
  int nstaged = 0, ngathered = 0, stage_bytes = 0, nstages = 0, nsplit = 1;
  int tiles_per_split = 0;
  int out_tma = 1;
  std::vector<int> leaf_stage_off;    // byte offset inside a stage, -1 = gathered
  int smem_bytes = 0, ctas_per_sm = 2;
};

constexpr int FG_FLAG_INTERPRET = 1 << 26;   // run group programs on the interpreter
constexpr int FG_FLAG_INJECT_NO_LOADS = 1 << 27;   // failure injection for tests
constexpr int FG_FLAG_NO_SMALL = 1 << 28;          // small groups too run the pipelined kernels

struct BuildOpts {
  int max_fused_ops = 256, max_args = 64, allow_reduce_epilogue = 0;
  int flags = 0;   // bits 8-15: tile band (GEMM: CTA-pair cap); see fg_build_opts in groupexec.h
  int64_t wait_limit_ns = 2000000000LL;
};

// Grouping (S1-S3).  Returns group_of[node] = sink node id and ipdom[node].
void partition(const Graph& g, const BuildOpts& o, std::vector<int32_t>& group_of,
               std::vector<int32_t>& ipdom);

// Group compilation (S4).  Throws CompileError on unsupported groups.
struct CompileError {
  fg_status st;
  std::string msg;
};
CompiledGroup compile_group(const Graph& g, const std::vector<int32_t>& nodes);
void plan_staging(const Graph& g, CompiledGroup& cg, const BuildOpts& o);

// Explicit fusion (host_explicit.cpp).  The partition owns a copy of the
// graph, which duplicate fusion extends with copies of operators (appended
// after the original nodes; their values are read only inside their group).
struct Partition {
  Graph g;
  std::vector<int32_t> label;      // per node: group label (the group's smallest node id)
  std::vector<int32_t> clone_of;   // per node: the copied operator, -1 for originals
  int max_fused_ops = 256;
};
// Throws CompileError when a group cannot run as one kernel.
using GroupCheck = std::function<void(const Graph&, const std::vector<int32_t>&)>;
Partition singleton_partition(const Graph& g, const BuildOpts& o);
// Fuses `node` with its predecessor `pred`; throws CompileError (FG_EINVAL,
// FG_EUNSUPPORTED) and leaves the partition unchanged when refused.
void fuse_move(Partition& P, int32_t node, int32_t pred, bool duplicate, const GroupCheck& check);
// Node lists of the groups in an order that respects their dependencies.
std::vector<std::vector<int32_t>> partition_groups(const Partition& P);
// Pattern-based grouping: chains of operators in priority order.
struct ChainPattern {
  std::vector<int32_t> ops;        // opcodes; ops[k+1] reads ops[k]'s output
  bool private_intermediates = false;
};
Partition pattern_partition(const Graph& g, const BuildOpts& o, const std::vector<ChainPattern>& pats,
                            const GroupCheck& check, std::vector<int32_t>& match_of);

}  // namespace fg
