/*
 * groupexec.h -- C ABI of libgroupexec.so: fused operator-group execution and
 * tensor-fusion pack/unpack on one GB300 (sm_103a).
 *
 * What is computed.
 *   A dataflow graph of operators is annotated with pattern kinds, a
 *   post-dominator tree is built on it, and operators are grouped by
 *   CheckPath/CommitFuse (TVM "Operator Fusion", Operator Pattern
 *   Classification; FuseOps > Algorithm, steps 1-4; Fusion rules).  Each
 *   group then runs as ONE kernel whose intermediates never reach device
 *   memory (DisCo, Introduction, on op fusion; TVM, FuseTIR: the merged
 *   function drops the intermediate buffers).  Separately, many small float32
 *   gradient tensors are scaled, cast and packed into one contiguous fusion
 *   buffer and unpacked again (DisCo, Introduction, on tensor fusion: the
 *   fused tensor's size is the sum of the parts).
 *
 * Conventions (all entry points).
 *   - Every function returns fg_status; FG_OK == 0.  On any other status a
 *     thread-local message is available from fg_last_error().
 *   - Ownership: the caller owns every tensor and the fusion buffer and passes
 *     raw DEVICE pointers (float32 or bfloat16, row-major, contiguous) and a
 *     CUDA stream as `void*` (NULL = legacy default stream).  The library owns
 *     graphs, plans and layouts and the small device tables they hold; it
 *     allocates device memory only in fg_build_groups / tf_layout_create,
 *     never in a launch, and frees it in the matching *_destroy.
 *   - Launches are asynchronous on the given stream.  Argument, shape and
 *     alignment errors are returned synchronously (tensors 16-byte aligned,
 *     fusion buffer 256-byte aligned).  CUDA launch errors map to FG_ECUDA.
 *     Errors found on the device (a bounded wait that expired) are latched in
 *     the plan's device flag and reported by fg_sync_status.
 *   - A plan is immutable after build.  Launches of one plan must be ordered:
 *     on one stream, or on streams ordered by events (each group owns small
 *     device state that a launch uses from start to end: the tile claim
 *     counter of an elementwise group, the split partials and arrival
 *     counters of a reduce group, the split workspace of a GEMM group).
 *     Plans are independent of each other: for concurrent launches, build one
 *     plan per stream (the compiled kernels are shared).
 *   - No CPU fallback exists: without a CUDA device every launch returns
 *     FG_ECUDA.  Graph building and grouping are host-only and work without a
 *     device.
 */
#ifndef GROUPEXEC_H
#define GROUPEXEC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FG_OK = 0,
  FG_EINVAL = 1,        /* bad argument: null pointer, unknown id, bad opcode */
  FG_ESHAPE = 2,        /* operand shapes do not fit the operator */
  FG_EUNSUPPORTED = 3,  /* valid graph the kernels cannot execute (reason in fg_last_error) */
  FG_ENOMEM = 4,        /* host or device allocation failed */
  FG_ECUDA = 5,         /* CUDA runtime/driver error, or no CUDA device */
  FG_ETIMEOUT = 6,      /* a device-side bounded wait expired */
  FG_EDEVICE = 7        /* other device-side error flag */
} fg_status;

typedef enum { FG_F32 = 0, FG_BF16 = 1 } fg_dtype;

/* Operators.  Kinds follow TVM's OpPatternKind (Operator Pattern
 * Classification): elementwise 0, broadcast 1, injective 2, commutative
 * reduce 3, out-elementwise-fusable 4, opaque 8.  All compute in float32 and
 * round after every operator; immediates are float32 attributes.
 *   ADD (2 or 3 operands, (a+b)+c), SUB, MUL, DIV         elementwise
 *   SCALE(imm) = imm*x, ADDC(imm) = x+imm, RELU (x>0?x:0),
 *   EXP, SIGMOID = 1/(1+exp(-x)), TANH, NEG               elementwise
 *   BADD_COL/BMUL_COL: x[R,C] (+|*) v[C]                   broadcast
 *   BADD_ROW/BMUL_ROW: x[R,C] (+|*) v[R]                   broadcast
 *   TRANSPOSE [R,C]->[C,R]; RESHAPE(rows, cols) row-major  injective
 *   ROWSUM, ROWMAX: [R,C] -> [R] over the last axis        commutative reduce
 *   MATMUL_BF16(transA, transB): bf16 x bf16 -> f32 [M,N]  out-elementwise-fusable
 *       A is [M,K] (or [K,M] when transA), B is [K,N] (or [N,K] when transB)
 *   OPAQUE_COPY: identity that never fuses                 opaque
 *   TUPLE(a, b[, c[, d]]): 2-D f32 fields of one width C; its value is the
 *       fields' rows stacked in order, [sum of rows, C]     tuple (7)
 *   CONCAT(t): joins the fields of tuple t (its only operand must be a
 *       TUPLE's value): [sum of rows, C]                     injective
 * A tuple fuses like an injective operator into its post-dominator (FuseOps
 * phase 1); phase 2 then fuses injective-or-simpler producers of its fields
 * into the group that absorbed it (TVM "Operator Fusion", Fusion rules).
 * Groups holding a tuple run compiled programs only.
 */
typedef enum {
  FG_OP_ADD = 0, FG_OP_SUB, FG_OP_MUL, FG_OP_DIV, FG_OP_SCALE, FG_OP_ADDC,
  FG_OP_RELU, FG_OP_EXP, FG_OP_SIGMOID, FG_OP_TANH, FG_OP_NEG,
  FG_OP_BADD_COL, FG_OP_BMUL_COL, FG_OP_BADD_ROW, FG_OP_BMUL_ROW,
  FG_OP_TRANSPOSE, FG_OP_RESHAPE, FG_OP_ROWSUM, FG_OP_ROWMAX,
  FG_OP_MATMUL_BF16, FG_OP_OPAQUE_COPY, FG_OP_TUPLE, FG_OP_CONCAT, FG_OP_COUNT
} fg_opcode;

/* Which kernel executes a group. */
typedef enum { FG_EXEC_ELEMWISE = 0, FG_EXEC_REDUCE = 1, FG_EXEC_GEMM = 2 } fg_exec_kind;

typedef struct fg_graph fg_graph;
typedef struct fg_plan fg_plan;
typedef struct tf_layout tf_layout;

/* Grouping options.  max_fused_ops: kMaxFusedOps (TVM, Fusion rules, the
 * constraints: 256).  max_args: the function-argument limit the page names
 * without a value; counts distinct outside values read plus one output.
 * allow_reduce_epilogue: let a reduce group absorb an elementwise tail on the
 * reduced vector (off = the page's rule that a reduction never fuses forward).
 * wait_limit_ns: bound on every device-side wait before it sets the error
 * flag and the kernel returns.  flags tune the kernels without changing
 * results: bits 8-15 = height in tiles of the bands the tile walk sweeps
 * column by column (0 = row-major walk), and for GEMM-epilogue groups the
 * most clusters to launch (0 = as many as the device runs at once); bits
 * 16-23 = tiles per reduce work unit (0 = chosen from the frame and the SM
 * count), and for GEMM-epilogue groups (which always run as CTA pairs;
 * bits 16-17 are ignored) bits 18-19 the K blocks of 64 per operand ring slot (0 = chosen,
 * 1, 2), bits 20-21 the schedule (0 = chosen, 1 = round robin with the last
 * round's tiles cut along K into two equal pieces, each finishing one column
 * half with the other's partial sums, the choice from 64 K blocks, 2 = equal
 * shares of all tiles' K steps, 3 = round robin with the last round's tiles
 * cut into their two column halves, the choice below 64 K blocks), bits 22-23
 * the columns of a CTA pair's tile (0 or 1 = 256, 2 = 128, 3 = 224); bits 24-25 = how an
 * elementwise group writes its output: 0 default (= 2), 1 the CTA's tile
 * staged in shared memory and stored by one TMA store, 2 each warp's slice
 * stored by its own TMA store, 3 direct 16-byte stores from registers; and
 * for GEMM-epilogue groups whose result is written in place of a leaf's
 * staged chunk, how it leaves (0 = chosen by K, 1 = the leaf producer's copy
 * of each 128 x 32 chunk before it reloads the buffer, 2 = each epilogue
 * warp's copy of its 32 rows; 3 = as 1); bits 29-30 the GEMM operand
 * ring's size (0 = chosen by K, 1 = 64 KB, 2 = 96 KB, 3 = 128 KB; the
 * epilogue's leaf buffers take the shared memory left, up to eight);
 * bit 28 turns off the direct kernel (groups of at most 2 MiB of leaves and
 * output whose frame rows hold at most 1024 elements, and row reductions of
 * at least 8192 row segments whose leaves are all read row by row,
 * otherwise run one warp per frame row segment, reading the leaves straight
 * from global memory, instead of the shared-memory pipeline);
 * bit 26 runs the groups' operator programs on the register-stack
 * interpreter instead of compiling each program to straight-line code when
 * the plan is built (default; needs NVRTC, loaded at run time); bit 27 is a
 * failure-injection hook for tests: the kernels' load producers issue
 * nothing, so every consumer's bounded wait expires and fg_sync_status
 * reports FG_ETIMEOUT with the context still usable. */
typedef struct {
  int32_t max_fused_ops;
  int32_t max_args;
  int32_t allow_reduce_epilogue;
  int32_t flags;
  int64_t wait_limit_ns;
} fg_build_opts;

/* Fills the defaults: 256, 64, 0, 0, 2e9 ns. */
void fg_build_opts_default(fg_build_opts* opts);

/* ---- graph construction (host only) ------------------------------------ */

/* New empty graph.  Value ids are assigned in creation order to inputs and
 * operator outputs alike; the i-th operator added is node i. */
fg_status fg_graph_create(fg_graph** g);

/* Graph input of rank 1 or 2.  bf16 inputs may only feed MATMUL_BF16. */
fg_status fg_graph_add_input(fg_graph* g, fg_dtype dtype, int32_t ndim,
                             const int64_t* shape, int32_t* value_id);

/* Operator over existing values (so the graph is topological by
 * construction).  attrs: SCALE/ADDC {imm}; RESHAPE {rows, cols};
 * MATMUL_BF16 {transA, transB}; others none.  Shapes are checked here
 * (FG_ESHAPE). */
fg_status fg_graph_add_op(fg_graph* g, int32_t opcode, int32_t n_in,
                          const int32_t* in_ids, int32_t n_attr,
                          const float* attrs, int32_t* value_id);

/* Marks a value as a graph output: it is always materialised. */
fg_status fg_graph_mark_output(fg_graph* g, int32_t value_id);

/* dtype, rank and shape (shape[1] = 1 for rank 1) of a value. */
fg_status fg_graph_value_info(const fg_graph* g, int32_t value_id, int32_t* dtype,
                              int32_t* ndim, int64_t* shape2);

void fg_graph_destroy(fg_graph* g);

/* ---- grouping and execution ---------------------------------------------- */

/* Annotate kinds, build the post-dominator tree, group (phases 0 and 1) and
 * compile each group into an operator program for its kernel.  Also compiles a
 * one-operator program per node for fg_launch_unfused.  Allocates the plan's
 * device error flag and reduce scratch when a CUDA device is present; without
 * one the plan is host-only (queries work, launches fail).  opts may be NULL
 * for the defaults.  A group the kernels cannot run (say a matmul operand
 * whose contiguous extent is not a multiple of 8, or a leaf that would be
 * gathered from a frame of 2^31 or more elements) does not fail the build:
 * the plan keeps the grouping, and that group's fg_plan_group_info (which
 * still fills its outputs), fg_plan_group_source and launches return its
 * status, FG_EUNSUPPORTED, with the reason in fg_last_error; the other
 * per-group diagnostics fill what they can and return FG_OK. */
fg_status fg_build_groups(const fg_graph* g, const fg_build_opts* opts, fg_plan** plan);

/* Node and group counts; group_of[node] = the node id of its group's sink
 * (largest node id in the group); ipdom[node] = immediate post-dominator
 * node or -1.  Either array may be NULL. */
fg_status fg_plan_query(const fg_plan* p, int32_t* n_nodes, int32_t* n_groups,
                        int32_t* group_of, int32_t* ipdom);

/* Group gid (0..n_groups-1, in order of sink node id).  Array outputs may be
 * NULL; `nodes` needs n_nodes entries and `leaves` n_leaves entries (call
 * once with NULL arrays to get the counts).  leaves are the value ids the
 * group reads from outside in first-use order; out_value is its one output;
 * kind is the fg_exec_kind; alg_bytes counts each leaf once plus the output;
 * alg_flops is 2*M*N*K for a GEMM group and 0 otherwise. */
fg_status fg_plan_group_info(const fg_plan* p, int32_t gid, int32_t* n_nodes,
                             int32_t* nodes, int32_t* n_leaves, int32_t* leaves,
                             int32_t* out_value, int32_t* kind,
                             int64_t* alg_bytes, int64_t* alg_flops);

/* Runs group gid as one kernel on `cuda_stream`.  value_ptrs is indexed by
 * value id and must hold device pointers for the group's leaves and output
 * (other entries are ignored and may be NULL). */
fg_status fg_launch_group(fg_plan* p, int32_t gid, void* const* value_ptrs, void* cuda_stream);

/* Runs one node on its own (the unfused baseline: its output is written to
 * device memory).  value_ptrs as above for that node's operands and output. */
fg_status fg_launch_unfused(fg_plan* p, int32_t node, void* const* value_ptrs, void* cuda_stream);

/* Synchronises the stream, then reads and clears the plan's device error flag:
 * FG_ETIMEOUT when a bounded wait expired, FG_EDEVICE for other flags.  On an
 * error it also zeroes the plan's split arrival counters, which a kernel that
 * gave up may have left mid-count, so the plan's next launches are correct;
 * results of the launches since the last FG_OK are undefined. */
fg_status fg_sync_status(fg_plan* p, void* cuda_stream);

/* Every value group gid writes: out_values[0] is the group's sink output
 * (the out_value of fg_plan_group_info), then its extra outputs: values
 * computed inside the group that operators outside it, or the caller, still
 * read (only explicit partitions make these; see fg_partition_fuse).
 * out_values: host, caller-owned, room for *n_out entries (query with NULL
 * first; at most 5). */
fg_status fg_plan_group_outputs(const fg_plan* p, int32_t gid, int32_t* n_out, int32_t* out_values);

/* Diagnostics for benchmarks: number of kernel launches fg_launch_group
 * issues for gid (always 1), the tile shape, pipeline depth and number of
 * TMA-staged leaves chosen for it. */
fg_status fg_plan_group_exec_info(const fg_plan* p, int32_t gid, int32_t* tile_rows,
                                  int32_t* tile_cols, int32_t* stages, int32_t* n_staged,
                                  int32_t* n_gathered, int32_t* prog_len);

/* Diagnostics: whether fg_launch_group runs gid on the direct kernel (leaves
 * read straight from global memory, one warp per frame row segment, no
 * shared-memory ring: small groups, and row reductions of at least 8192 row
 * segments whose leaves are all read row by row), the warps per frame row
 * (1 unless direct), and whether its launch always may begin while the
 * stream's previous kernel finishes (a large direct launch does so only
 * behind another direct launch).  Any output pointer may be NULL.  Host
 * only; FG_EINVAL for a null plan or an unknown group. */
fg_status fg_plan_group_direct_info(const fg_plan* p, int32_t gid, int32_t* direct, int32_t* segments,
                                    int32_t* early_launch);

/* The CUDA source the plan compiles for group gid (the group's operator
 * program written out as straight-line code inside the shared pipeline).
 * Writes at most cap bytes including the terminating NUL to buf (buf may be
 * NULL) and the full length without the NUL to *len_out. */
fg_status fg_plan_group_source(const fg_plan* p, int32_t gid, char* buf, int64_t cap, int64_t* len_out);

void fg_plan_destroy(fg_plan* p);

/* Message for the last non-OK status on this thread ("" if none). */
const char* fg_last_error(void);

/* Row reduction without device allocation: y[r] = sum over c of x[r, c]
 * (opcode FG_OP_ROWSUM) or the maximum over c (FG_OP_ROWMAX) of a row-major
 * float32 matrix x[rows, cols], for callers that cannot call cudaMalloc -- a
 * host framework that owns every device allocation through its own pool, or
 * a step that cannot accept the device-wide synchronisation an allocation
 * may imply -- and so cannot build a plan either.  The pages have no
 * counterpart of this entry point.  It runs the reduce-group kernel on a
 * one-operator program with its scratch (per-split partial row values and
 * arrival counters, and an error word) in a file-scope device array of
 * 4 MiB + 8 KiB + 256 bytes that every
 * GPU which loads the library holds until the process exits.
 * Limits: rows <= 65536 (else FG_EINVAL) and rows*cols < 2^31 (else
 * FG_ESHAPE).  x (16-byte aligned) and y (4-byte aligned) are device
 * pointers owned by the caller.  Asynchronous on cuda_stream.  The first
 * call on a device (and on each host thread with no current context, and
 * the first after the device's context was created again) looks up the
 * array's device address; make that call before any stream capture.  All
 * calls share the array, so calls that overlap on the GPU (other streams,
 * or host threads without ordering) race.  A bounded device-side wait (2 s)
 * that expires latches an error word in the same array and leaves y
 * incomplete; the call itself cannot see it (it returns before the kernel
 * runs): fg_row_reduce_noalloc_status reports it. */
fg_status fg_row_reduce_noalloc(int32_t opcode, const float* x, int64_t rows, int64_t cols, float* y,
                                void* cuda_stream);

/* Synchronizes cuda_stream, then reads and clears the error word that
 * fg_row_reduce_noalloc's kernels latch on the current device: FG_OK if no
 * call since the last read gave up, FG_ETIMEOUT if a bounded wait expired
 * (that call's y is incomplete), FG_ECUDA for a CUDA error.  Allocates
 * nothing.  No counterpart on the pages either. */
fg_status fg_row_reduce_noalloc_status(void* cuda_stream);

/* ---- explicit fusion --------------------------------------------------------
 * DisCo, Introduction and Strategy Maker, optimisation methods (i) and (ii):
 * an operator is fused with one of the predecessors whose output it reads.
 * When that predecessor has other readers, non-duplicate fusion folds it into
 * the fused group, whose output then also serves those readers (the group
 * gains an extra output), while duplicate fusion puts a copy of it into the
 * group and keeps the original for its other readers.  The search that
 * chooses the moves is the caller's. */
typedef struct fg_partition fg_partition;

/* A partition of g's operators: every operator alone (from_fuseops = 0) or the
 * FuseOps grouping of fg_build_groups (from_fuseops = 1).  The partition keeps
 * its own copy of the graph; opts as for fg_build_groups (max_fused_ops and
 * max_args bound every fused group). */
fg_status fg_partition_create(const fg_graph* g, const fg_build_opts* opts, int32_t from_fuseops,
                              fg_partition** out);

/* Fuses operator `node` with operator `pred`, whose output must be an
 * operand of `node`; duplicate = 1 for duplicate fusion (a predecessor that
 * nothing else reads is simply merged either way).  Duplicate fusion appends
 * a copy of `pred` to the partition's graph (node id = the old node count,
 * its value id = the old value count; its value is never materialised).
 * Returns FG_EINVAL (not a predecessor, already one group, bad id) or
 * FG_EUNSUPPORTED (the merged group would not be convex, or would not run as
 * one kernel: two reductions, a matmul with extra outputs, more than 4 extra
 * outputs, an extra output after a reduction or without the frame's element
 * count, or the max_fused_ops / max_args bounds); the partition is then
 * unchanged. */
fg_status fg_partition_fuse(fg_partition* p, int32_t node, int32_t pred, int32_t duplicate);

/* Pattern-based grouping (TVM "Operator Fusion", FuseOpsByPattern): the
 * caller names which operator combinations form groups.  A pattern is a chain
 * of operators, each reading the previous one's output (as any operand; other
 * operands are wildcards).  Anchors are tried in node order and, at each, the
 * patterns in the given (priority) order; the chain's next operator is the
 * smallest-numbered reader of the previous output with the pattern's opcode
 * that no earlier match took.  A match is kept only if it is convex, passes
 * the private check when private_intermediates = 1 (no intermediate result
 * read outside the match or marked as a graph output) and runs as one kernel
 * (as fg_partition_fuse checks); every other operator stays alone.  The
 * partition can then be changed with fg_partition_fuse and built with
 * fg_build_from_partition.  match_of: host, caller-owned, one entry per
 * operator (the pattern index, or -1), or NULL. */
typedef struct {
  int32_t n_ops;
  const int32_t* opcodes;           /* fg_opcode values, chain order */
  int32_t private_intermediates;
} fg_pattern;
fg_status fg_partition_from_patterns(const fg_graph* g, const fg_build_opts* opts, int32_t n_patterns,
                                     const fg_pattern* patterns, fg_partition** out, int32_t* match_of);

/* n_nodes: operators including copies; group_of[i]: the group's smallest node
 * id; clone_of[i]: the operator node i copies, -1 for originals.  Arrays are
 * host, caller-owned, n_nodes entries, or NULL. */
fg_status fg_partition_query(const fg_partition* p, int32_t* n_nodes, int32_t* group_of, int32_t* clone_of);

/* A plan for the partition's groups (same queries and launches as a
 * fg_build_groups plan).  Group ids follow a dependency order: launching
 * groups 0, 1, ... computes every output.  fg_plan_query reports the
 * partition's labels as group_of and -1 as ipdom.  Extra outputs need a
 * pointer in value_ptrs like any output; groups with extra outputs run
 * compiled programs only. */
fg_status fg_build_from_partition(const fg_partition* p, fg_plan** plan);

void fg_partition_destroy(fg_partition* p);

/* ---- training-step simulator ----------------------------------------------
 * DisCo, Simulator: computation operators (e.g. the groups of a plan, with
 * measured times) run one at a time from a FIFO ready queue: the queue
 * starts with the operators without dependencies in index order, and an
 * operator joins its tail when its last dependency clears (successors in
 * index order).  AllReduce instructions (one per bucket of gradient tensors)
 * run on one channel in the order their buckets are complete (ties in bucket
 * order), each once every tensor it carries is produced and the channel is
 * free, overlapping with computation; one of x bytes takes ar_c * x + ar_d
 * (DisCo, Profiler; a ring over N devices with narrowest link bandwidth B has
 * ar_c = 2(N-1)/(B*N)).  An operator may wait for AllReduces (ar edges): it
 * joins the queue once they are scheduled and starts at their completion at
 * the earliest.  All arrays are host and caller-owned; times and bytes in the
 * caller's units. */
typedef struct {
  int32_t n_ops;
  const double* op_time;            /* [n_ops] */
  int32_t n_edges;
  const int32_t* edge_src;          /* [n_edges] operator edge_src[e] before edge_dst[e] */
  const int32_t* edge_dst;
  int32_t n_tensors;
  const int32_t* tensor_producer;   /* [n_tensors] operator that produces each gradient tensor */
  const double* tensor_bytes;       /* [n_tensors] */
  int32_t n_buckets;
  const int32_t* bucket_bounds;     /* [n_buckets + 1] ranges of bucket_tensors */
  const int32_t* bucket_tensors;    /* tensor ids, bucket after bucket */
  double ar_c, ar_d;
  int32_t n_ar_edges;
  const int32_t* ar_edge_bucket;    /* [n_ar_edges] operator ar_edge_op[e] waits for bucket ar_edge_bucket[e] */
  const int32_t* ar_edge_op;
} fg_sim_problem;

/* *total: the time the last operator or AllReduce completes; op_finish
 * [n_ops], ar_start / ar_finish [n_buckets]: optional outputs (NULL to skip).
 * FG_EINVAL on out-of-range ids, bad bounds or a dependency cycle.  Host
 * only. */
fg_status fg_simulate(const fg_sim_problem* p, double* total, double* op_finish, double* ar_start,
                      double* ar_finish);

/* ---- tensor fusion ------------------------------------------------------- */

/* The layout of tf_layout_create computed on the host alone (no device, no
 * allocation): offsets_out[i] (n entries, or NULL) and total_bytes_out (or
 * NULL).  For allocating the fusion buffer before the layout exists, or for
 * a peer that only needs the byte ranges.  FG_EINVAL / FG_ESHAPE as
 * tf_layout_create. */
fg_status tf_layout_offsets(int32_t n, const int64_t* numel, fg_dtype buf_dtype, int64_t align_bytes,
                            int64_t* offsets_out, int64_t* total_bytes_out);

/* Layout of n float32 gradient tensors (device pointers grads[i], numel[i]
 * elements, 16-byte aligned) in one fusion buffer of buf_dtype (FG_BF16 or
 * FG_F32): tensor i starts at byte offset offsets_out[i], a multiple of
 * align_bytes (a power of two >= 16; 256 recommended); tensors are in index
 * order; total_bytes_out is the end of the last tensor rounded up to
 * align_bytes.  Uploads a chunk table to the device (requires a device). */
fg_status tf_layout_create(int32_t n, const int64_t* numel, float* const* grads,
                           fg_dtype buf_dtype, int64_t align_bytes, tf_layout** out,
                           int64_t* offsets_out, int64_t* total_bytes_out);

/* One kernel: buf[offset_i + k] = cast(fp32(grads[i][k] * scale)) with
 * round-to-nearest-even for bf16, and every padding byte set to 0.
 * fusion_buf: device, 256-byte aligned, at least total_bytes. */
fg_status tf_pack(const tf_layout* l, float scale, void* fusion_buf, void* cuda_stream);

/* One kernel: grads[i][k] = fp32(widen(buf[offset_i + k]) * uscale).
 * fusion_buf: device, 256-byte aligned.  The kernel waits (at most 100 ms
 * each) for its own chunk loads; an expired wait is recorded on the device
 * and reported by tf_sync_status. */
fg_status tf_unpack(const tf_layout* l, float uscale, const void* fusion_buf, void* cuda_stream);

/* Synchronises cuda_stream and returns FG_ETIMEOUT (clearing the record) if a
 * tf_unpack since the last call recorded an expired wait, else FG_OK. */
fg_status tf_sync_status(tf_layout* l, void* cuda_stream);

/* ---- AllReduce buckets ----------------------------------------------------
 * A bucket is a contiguous run of tensors (production order) whose bytes in
 * the fusion buffer form one fused AllReduce tensor: bucket b holds tensors
 * bounds[b] .. bounds[b+1]-1 and spans bytes offsets[bounds[b]] up to the
 * next bucket's start (or total_bytes).  DisCo, Related Work (Horovod's
 * fusion threshold, like XLA's AllReduce combiner) and Strategy Maker,
 * optimisation method (iii) (combining an AllReduce with a neighbour). */

/* Threshold fusion: greedy in tensor order, a tensor joins the open bucket
 * while the bucket's bytes (each tensor's numel * elem bytes rounded up to
 * align_bytes) stay <= threshold_bytes, else it opens the next bucket, so a
 * tensor above the threshold sits alone.  bounds: host, n + 1 entries
 * (caller-owned); *n_buckets receives the bucket count (0 when n == 0).
 * Host only: needs no device. */
fg_status tf_plan_threshold(int32_t n, const int64_t* numel, fg_dtype buf_dtype,
                            int64_t align_bytes, int64_t threshold_bytes,
                            int32_t* bounds, int32_t* n_buckets);

/* Neighbour combination: bucket j absorbs bucket j+1 (bounds and *n_buckets
 * updated in place).  FG_EINVAL if j has no successor.  Host only. */
fg_status tf_buckets_merge(int32_t* bounds, int32_t* n_buckets, int32_t j);

/* tf_pack / tf_unpack restricted to tensors first .. first+count-1 (one
 * launch; e.g. one bucket, as soon as its gradients exist).  Bytes outside
 * those tensors' ranges (data and padding) are not touched.  FG_EINVAL if
 * the range exceeds the layout. */
fg_status tf_pack_range(const tf_layout* l, int32_t first, int32_t count, float scale,
                        void* fusion_buf, void* cuda_stream);
fg_status tf_unpack_range(const tf_layout* l, int32_t first, int32_t count, float uscale,
                          const void* fusion_buf, void* cuda_stream);

/* One-launch packing of AllReduce buckets (DisCo, Introduction: each fused
 * buffer's AllReduce starts once its tensors are in it).
 *
 * tf_layout_set_buckets: the bucket table, bounds[0 .. n_buckets] as
 * tf_plan_threshold writes it (bounds[0] = 0, strictly increasing,
 * bounds[n_buckets] = the layout's tensor count; host, caller-owned, copied).
 * Replaces an earlier table without synchronizing: the old table stays
 * allocated until the events recorded after every pack and stream wait that
 * read it have completed (checked at the next replacement, waited for by
 * tf_layout_destroy).  Allocates the per-bucket device counts of written
 * chunks (zero) and restarts the launch numbering, so call it between steps:
 * a wait enqueued afterwards refers to the new table.  FG_EINVAL for a
 * malformed table.
 *
 * tf_pack_buckets: packs every tensor in one launch, with tf_pack's result,
 * and counts every chunk written for its bucket (a release reduction at GPU
 * scope, after the chunk's bytes, into a count that is never reset): bucket
 * b of the k-th launch since the table was set is complete, all its bytes
 * visible, once its count reaches k times its chunk count (compared
 * cyclically: the count wraps modulo 2^32).  FG_EINVAL without a bucket
 * table.
 *
 * tf_bucket_wait: makes cuda_stream wait, in the GPU's front end (no kernel,
 * no SM), until bucket b of the most recently enqueued tf_pack_buckets launch
 * is ready; work enqueued on that stream afterwards (the bucket's AllReduce)
 * reads its bytes.  The pack launch must already be enqueued (on any stream
 * that does not itself wait for cuda_stream): FG_EINVAL if none is, or if b
 * is out of range.
 *
 * tf_bucket_ready: *ready = 1 if bucket b of the most recently enqueued
 * tf_pack_buckets launch is complete, else 0 (a synchronous read of the
 * bucket's count; host-side polling).  The read is a cudaMemcpy
 * on the legacy default stream, so it also waits for work on that stream
 * and on every blocking stream: to watch a pack while it runs, enqueue the
 * pack on a non-blocking stream (PyTorch's side streams are).  FG_EINVAL as
 * for tf_bucket_wait.  Launches of one layout must be ordered (one stream, or
 * streams that wait for each other): they share the bucket counts. */
fg_status tf_layout_set_buckets(tf_layout* l, int32_t n_buckets, const int32_t* bounds);
fg_status tf_pack_buckets(tf_layout* l, float scale, void* fusion_buf, void* cuda_stream);
fg_status tf_bucket_wait(tf_layout* l, int32_t bucket, void* cuda_stream);
fg_status tf_bucket_ready(const tf_layout* l, int32_t bucket, int32_t* ready);

/* tf_pack_buckets with a device-side consumer of the bucket counts inside
 * the same launch (DisCo, Introduction: a bucket's AllReduce can start as
 * soon as its tensors are in the fusion buffer; a collective's own kernel
 * would watch the counts this way).  One extra CTA of the launch packs
 * nothing: it reads each bucket's count in bucket order (acquire, polled)
 * until it reaches the total of the launch seq_offset launches after this
 * one (0: this one), and writes the
 * device's global timer (ns) at that moment to times[b]; the packing CTAs
 * write the latest time any of them finished to times[n_buckets].  times:
 * device, 8-byte aligned, n_buckets + 1 entries, caller-owned.  Each wait is
 * bounded by wait_limit_ns: a wait that expires leaves times[b] = 0 for that
 * bucket and the rest, and latches FG_ETIMEOUT for tf_sync_status (a test
 * passes seq_offset = 1, a launch that never comes, to see that happen; use
 * 0 otherwise).  The fusion buffer receives exactly tf_pack_buckets' bytes.
 * One CTA watching and the others packing are one launch, so the watcher
 * never waits for work that cannot be scheduled. */
fg_status tf_pack_buckets_observed(tf_layout* l, float scale, void* fusion_buf, uint64_t* times,
                                   uint32_t seq_offset, int64_t wait_limit_ns, void* cuda_stream);

void tf_layout_destroy(tf_layout* l);

#ifdef __cplusplus
}
#endif

#endif /* GROUPEXEC_H */
