// The C ABI (include/groupexec.h): graph construction, grouping, plan
// queries, group launches and tensor-fusion layouts.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "host.h"
#include "jit.h"
#include "launch.h"

using namespace fg;

// ---------------------------------------------------------------------------
// errors
namespace {
thread_local std::string g_last_error;

fg_status err(fg_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}
fg_status cuda_err(cudaError_t e, const char* what) {
  return err(FG_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library loads on machines without a driver.
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn encode_fn() {
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

bool device_present(int* nsm) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
    cudaGetLastError();
    return false;
  }
  int dev = 0;
  cudaGetDevice(&dev);
  if (nsm) cudaDeviceGetAttribute(nsm, cudaDevAttrMultiProcessorCount, dev);
  return true;
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
}  // namespace

namespace fg {
int set_last_error(int status, const char* msg) { return err(static_cast<fg_status>(status), msg); }
}  // namespace fg

// ---------------------------------------------------------------------------
// opaque handles
struct fg_graph {
  Graph g;
};

namespace {
struct GroupExec {
  CompiledGroup cg;
  std::unique_ptr<GroupParams> gp;   // K1 / K2
  std::unique_ptr<GemmParams> mp;    // K3
  bool big = false;
  int grid = 1, smem = 0;
  float* scratch = nullptr;
  int32_t* counters = nullptr;        // split arrival counters (zero between launches)
  unsigned long long* sched = nullptr;   // K1 tile claim counter (see the kernel)
  size_t counter_bytes = 0;
  std::string compile_error;          // non-empty: cannot launch
  fg_status compile_status = FG_OK;
  bool compiled = false;              // run the compiled program (else the interpreter)
  int min_blocks = 2;                 // CTAs per SM the kernel is built for
  void* fn = nullptr;                 // compiled kernel
  bool small = false;                 // run the direct kernel instead (direct reads, no ring)
  bool small_pdl = true;              // ... launched early behind the stream's previous kernel
  int grid_small = 1;
  void* fn_small = nullptr;
  std::vector<const void*> last_ptrs; // tensor-map cache key
};
}  // namespace

struct fg_plan {
  Graph g;
  BuildOpts opts;
  std::vector<int32_t> group_of, ipdom;
  std::vector<GroupExec> groups;     // by gid (ascending sink)
  std::vector<GroupExec> singles;    // per node, for fg_launch_unfused
  bool has_device = false;
  int nsm = 148;
  int32_t* d_err = nullptr;
};

struct fg_partition {
  Partition P;
  BuildOpts opts;
};

struct tf_layout {
  int32_t n = 0;
  int buf_bf16 = 1;
  int64_t total = 0;
  std::vector<int64_t> numel, offsets;
  std::vector<float*> grads;
  TfChunk* d_chunks = nullptr;       // chunk table, followed by the device error word
  int32_t* d_err = nullptr;
  // chunk claim counter of packs over the whole layout (each launch
  // advances it by the chunk count)
  unsigned long long* d_claim = nullptr;
  int nchunks = 0;
  std::vector<int32_t> chunk_begin;  // first chunk of every tensor, [n + 1]
  // AllReduce buckets packed in one launch: device block of the chunk ->
  // bucket map [nchunks], chunks per bucket [nb] and counts [nb] (chunks
  // written by every bucketed pack so far, never reset); seq = the number of
  // bucketed packs enqueued with this table: bucket b of the last one is
  // complete once its count reaches seq * bucket_chunks[b]
  int32_t nb = 0;
  int32_t* d_bucket = nullptr;
  uint32_t seq = 0;
  std::vector<uint32_t> bucket_chunks;
  // the table's users: per stream, an event recorded after the last pack or
  // stream wait enqueued there that reads the table
  std::vector<std::pair<cudaStream_t, cudaEvent_t>> users;
  // tables replaced while a launch or wait might still read them, freed once
  // their users' events have completed
  struct Retired {
    int32_t* table;
    std::vector<std::pair<cudaStream_t, cudaEvent_t>> users;
  };
  std::vector<Retired> retired;
};

namespace {
// Records on `st` that the current bucket table is read by work enqueued
// there (one event per stream, re-recorded).
cudaError_t note_table_use(tf_layout* l, cudaStream_t st) {
  for (auto& u : l->users)
    if (u.first == st) return cudaEventRecord(u.second, st);
  cudaEvent_t ev;
  cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return e;
  l->users.emplace_back(st, ev);
  return cudaEventRecord(ev, st);
}

// Frees the replaced tables whose users have all finished (wait = block
// until they have).
void free_retired(tf_layout* l, bool wait) {
  std::vector<tf_layout::Retired> keep;
  for (auto& r : l->retired) {
    bool done = true;
    for (auto& u : r.users) {
      const cudaError_t q = wait ? cudaEventSynchronize(u.second) : cudaEventQuery(u.second);
      if (q == cudaErrorNotReady) done = false;
    }
    if (!done) {
      keep.push_back(std::move(r));
      continue;
    }
    for (auto& u : r.users) cudaEventDestroy(u.second);
    cudaFree(r.table);
  }
  l->retired.swap(keep);
  cudaGetLastError();   // a not-ready query is not an error of the caller's
}
}  // namespace

// cuStreamWaitValue32 through the runtime's driver entry point (no link
// against the driver library).
using WaitValueFn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
WaitValueFn wait_value_fn() {
  static WaitValueFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WaitValueFn>(p);
  });
  return fn;
}

// ---------------------------------------------------------------------------
extern "C" {

const char* fg_last_error(void) { return g_last_error.c_str(); }

void fg_build_opts_default(fg_build_opts* o) {
  if (!o) return;
  o->max_fused_ops = 256;
  o->max_args = 64;
  o->allow_reduce_epilogue = 0;
  o->flags = 0;
  o->wait_limit_ns = 2000000000LL;
}

fg_status fg_graph_create(fg_graph** g) {
  if (!g) return err(FG_EINVAL, "null output pointer");
  *g = new (std::nothrow) fg_graph();
  return *g ? FG_OK : err(FG_ENOMEM, "out of host memory");
}

void fg_graph_destroy(fg_graph* g) { delete g; }

fg_status fg_graph_add_input(fg_graph* gh, fg_dtype dtype, int32_t ndim, const int64_t* shape, int32_t* vid) {
  if (!gh || !shape || !vid) return err(FG_EINVAL, "null argument");
  if (dtype != FG_F32 && dtype != FG_BF16) return err(FG_EINVAL, "unknown dtype");
  if (ndim != 1 && ndim != 2) return err(FG_ESHAPE, "inputs have rank 1 or 2");
  Value v;
  v.dtype = dtype;
  v.ndim = ndim;
  v.rows = ndim == 2 ? shape[0] : 1;
  v.cols = ndim == 2 ? shape[1] : shape[0];
  if (v.rows <= 0 || v.cols <= 0) return err(FG_ESHAPE, "empty or negative extent");
  if (v.rows > (int64_t(1) << 31) - 64 || v.cols > (int64_t(1) << 31) - 64) return err(FG_ESHAPE, "extent too large");
  v.is_input = true;
  gh->g.values.push_back(v);
  gh->g.is_output.push_back(0);
  *vid = (int32_t)gh->g.values.size() - 1;
  return FG_OK;
}

fg_status fg_graph_add_op(fg_graph* gh, int32_t op, int32_t n_in, const int32_t* in_ids, int32_t n_attr,
                          const float* attrs, int32_t* vid) {
  if (!gh || !vid || (n_in > 0 && !in_ids) || (n_attr > 0 && !attrs)) return err(FG_EINVAL, "null argument");
  if (op < 0 || op >= FG_OP_COUNT) return err(FG_EINVAL, "unknown opcode");
  Graph& g = gh->g;
  for (int i = 0; i < n_in; ++i)
    if (in_ids[i] < 0 || in_ids[i] >= (int32_t)g.values.size()) return err(FG_EINVAL, "unknown operand value id");
  auto need = [&](int lo, int hi, int na) -> fg_status {
    if (n_in < lo || n_in > hi) return err(FG_EINVAL, "wrong number of operands");
    if (n_attr < na) return err(FG_EINVAL, "missing attribute");
    return FG_OK;
  };
  auto V = [&](int i) -> const Value& { return g.values[in_ids[i]]; };
  Value out;
  out.is_input = false;
  fg_status st = FG_OK;
  switch (op) {
    case FG_OP_ADD:
      if ((st = need(2, 3, 0))) return st;
      for (int i = 1; i < n_in; ++i) if (!V(i).same_shape(V(0))) return err(FG_ESHAPE, "add operands differ in shape");
      out = V(0);
      break;
    case FG_OP_SUB: case FG_OP_MUL: case FG_OP_DIV:
      if ((st = need(2, 2, 0))) return st;
      if (!V(1).same_shape(V(0))) return err(FG_ESHAPE, "operands differ in shape");
      out = V(0);
      break;
    case FG_OP_SCALE: case FG_OP_ADDC:
      if ((st = need(1, 1, 1))) return st;
      out = V(0);
      break;
    case FG_OP_RELU: case FG_OP_EXP: case FG_OP_SIGMOID: case FG_OP_TANH: case FG_OP_NEG: case FG_OP_OPAQUE_COPY:
      if ((st = need(1, 1, 0))) return st;
      out = V(0);
      break;
    case FG_OP_BADD_COL: case FG_OP_BMUL_COL: case FG_OP_BADD_ROW: case FG_OP_BMUL_ROW: {
      if ((st = need(2, 2, 0))) return st;
      bool col = op == FG_OP_BADD_COL || op == FG_OP_BMUL_COL;
      if (V(0).ndim != 2 || V(1).ndim != 1 || V(1).cols != (col ? V(0).cols : V(0).rows))
        return err(FG_ESHAPE, "broadcast needs x[R,C] and a vector of length C (col) or R (row)");
      out = V(0);
      break;
    }
    case FG_OP_TRANSPOSE:
      if ((st = need(1, 1, 0))) return st;
      if (V(0).ndim != 2) return err(FG_ESHAPE, "transpose needs rank 2");
      out = V(0);
      std::swap(out.rows, out.cols);
      break;
    case FG_OP_RESHAPE: {
      if ((st = need(1, 1, 2))) return st;
      int64_t r = (int64_t)attrs[0], c = (int64_t)attrs[1];
      if (r <= 0 || c <= 0 || r * c != V(0).numel()) return err(FG_ESHAPE, "reshape must keep the element count");
      out = V(0);
      out.ndim = 2;
      out.rows = r;
      out.cols = c;
      break;
    }
    case FG_OP_ROWSUM: case FG_OP_ROWMAX:
      if ((st = need(1, 1, 0))) return st;
      if (V(0).ndim != 2) return err(FG_ESHAPE, "row reduction needs rank 2");
      out = V(0);
      out.ndim = 1;
      out.cols = V(0).rows;
      out.rows = 1;
      break;
    case FG_OP_TUPLE: {
      if ((st = need(2, 4, 0))) return st;
      int64_t rows = 0;
      for (int i = 0; i < n_in; ++i) {
        if (V(i).ndim != 2) return err(FG_ESHAPE, "tuple fields must be rank-2");
        if (V(i).cols != V(0).cols) return err(FG_ESHAPE, "tuple fields must have one width");
        if (V(i).node >= 0 && g.nodes[V(i).node].op == FG_OP_TUPLE) return err(FG_EUNSUPPORTED, "a tuple of tuples");
        rows += V(i).rows;
      }
      out.ndim = 2;
      out.rows = rows;
      out.cols = V(0).cols;
      break;
    }
    case FG_OP_CONCAT:
      if ((st = need(1, 1, 0))) return st;
      if (V(0).node < 0 || g.nodes[V(0).node].op != FG_OP_TUPLE)
        return err(FG_EINVAL, "concat reads the value of a tuple");
      out.ndim = 2;
      out.rows = V(0).rows;
      out.cols = V(0).cols;
      break;
    case FG_OP_MATMUL_BF16: {
      if ((st = need(2, 2, 0))) return st;
      int ta = n_attr > 0 ? (int)attrs[0] : 0, tb = n_attr > 1 ? (int)attrs[1] : 0;
      const Value &A = V(0), &B = V(1);
      if (A.dtype != FG_BF16 || B.dtype != FG_BF16) return err(FG_EINVAL, "matmul operands must be bf16");
      if (A.ndim != 2 || B.ndim != 2) return err(FG_ESHAPE, "matmul needs rank-2 operands");
      int64_t M = ta ? A.cols : A.rows, KA = ta ? A.rows : A.cols;
      int64_t KB = tb ? B.cols : B.rows, N = tb ? B.rows : B.cols;
      if (KA != KB) return err(FG_ESHAPE, "matmul inner extents differ");
      out.ndim = 2;
      out.rows = M;
      out.cols = N;
      break;
    }
    default:
      return err(FG_EINVAL, "unknown opcode");
  }
  if (op != FG_OP_MATMUL_BF16) {
    for (int i = 0; i < n_in; ++i)
      if (V(i).dtype != FG_F32) return err(FG_EUNSUPPORTED, "bf16 values can only feed MATMUL_BF16");
  }
  out.dtype = FG_F32;
  out.is_input = false;
  Node n;
  n.op = op;
  n.args.assign(in_ids, in_ids + n_in);
  if (n_attr > 0) n.attrs.assign(attrs, attrs + n_attr);
  out.node = (int32_t)g.nodes.size();
  n.value = (int32_t)g.values.size();
  g.values.push_back(out);
  g.is_output.push_back(0);
  g.nodes.push_back(n);
  *vid = n.value;
  return FG_OK;
}

fg_status fg_graph_mark_output(fg_graph* gh, int32_t vid) {
  if (!gh) return err(FG_EINVAL, "null graph");
  if (vid < 0 || vid >= (int32_t)gh->g.values.size()) return err(FG_EINVAL, "unknown value id");
  gh->g.is_output[vid] = 1;
  return FG_OK;
}

fg_status fg_graph_value_info(const fg_graph* gh, int32_t vid, int32_t* dtype, int32_t* ndim, int64_t* shape2) {
  if (!gh) return err(FG_EINVAL, "null graph");
  if (vid < 0 || vid >= (int32_t)gh->g.values.size()) return err(FG_EINVAL, "unknown value id");
  const Value& v = gh->g.values[vid];
  if (dtype) *dtype = v.dtype;
  if (ndim) *ndim = v.ndim;
  if (shape2) {
    shape2[0] = v.ndim == 2 ? v.rows : v.cols;
    shape2[1] = v.ndim == 2 ? v.cols : 1;
  }
  return FG_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// plan construction
namespace {

void fill_leaf_desc(LeafDesc& d, const LeafUse& l, int stage_off, int map_idx, int64_t FC) {
  std::memset(&d, 0, sizeof(d));
  d.cls = l.cls;
  d.stage_off = stage_off;
  d.map_idx = map_idx;
  d.shift = l.map.shift;
  d.numel = l.numel;
  d.shift_r = (int32_t)(l.map.shift / FC);
  d.shift_c = (int32_t)(l.map.shift % FC);
  d.nterms = l.map.n;
  for (int k = 0; k < l.map.n; ++k) {
    d.d[k] = l.map.d[k];
    d.m[k] = l.map.m[k];
    d.s[k] = l.map.s[k];
    d.dd[k] = fast_div(l.map.d[k]);
    d.dm[k] = fast_div(l.map.m[k]);
  }
}

int box_tx_bytes(int cls) {
  switch (cls) {
    case LEAF_IDENT: case LEAF_TRANS: return kTileR * kTileC * 4;
    case LEAF_COL: return kTileC * 4;
    case LEAF_ROW: return kTileR * 4;
    default: return 0;
  }
}

// Static part of the kernel parameters of a K1/K2 group.
void prepare_group(GroupExec& ge, const BuildOpts& o, int nsm) {
  CompiledGroup& cg = ge.cg;
  ge.gp.reset(new GroupParams());
  GroupParams& p = *ge.gp;
  std::memset(&p, 0, sizeof(p));
  if (cg.prog.size() > (size_t)kMaxProg) throw CompileError{FG_EUNSUPPORTED, "group program too long"};
  std::copy(cg.prog.begin(), cg.prog.end(), p.prog);
  p.nprog = (int)cg.prog.size();
  p.nleaves = (int)cg.leaves.size();
  int mi = 0, tx = 0;
  for (size_t i = 0; i < cg.leaves.size(); ++i) {
    bool staged = cg.leaves[i].cls != LEAF_GATHER;
    fill_leaf_desc(p.leaves[i], cg.leaves[i], staged ? cg.leaf_stage_off[i] : -1, staged ? mi : -1, cg.FC);
    if (staged) {
      ++mi;
      tx += box_tx_bytes(cg.leaves[i].cls);
    }
  }
  p.nstaged = mi;
  p.nxout = (int32_t)cg.xout_values.size();
  p.xout_tma = cg.xout_tma;
  for (int j = 0; j < p.nxout; ++j) {
    const Map& mp = cg.xout_maps[j];
    XOutDesc& x = p.xout[j];
    x.cls = cg.xout_cls[j];
    x.nterms = mp.n;
    for (int k = 0; k < mp.n; ++k) {
      x.d[k] = mp.d[k];
      x.m[k] = mp.m[k];
      x.s[k] = mp.s[k];
      x.dd[k] = fast_div(mp.d[k]);
      x.dm[k] = fast_div(mp.m[k]);
    }
  }
  std::copy(cg.epi.begin(), cg.epi.end(), p.epi);
  p.nepi = (int)cg.epi.size();
  p.FR = (int32_t)cg.FR;
  p.FC = (int32_t)cg.FC;
  p.ntr = (int32_t)((cg.FR + kTileR - 1) / kTileR);
  p.ntc = (int32_t)((cg.FC + kTileC - 1) / kTileC);
  p.ntiles = p.ntr * p.ntc;
  p.stage_bytes = cg.stage_bytes;
  p.nstages = cg.nstages;
  p.tx_bytes = tx;
  p.out_tma = cg.out_tma;
  p.band = (o.flags >> 8) & 0xff;
  p.inject = (o.flags & FG_FLAG_INJECT_NO_LOADS) ? 1 : 0;
  p.wait_limit_ns = o.wait_limit_ns;
  ge.big = std::max(cg.depth, cg.epi_depth) > 4 || std::max(cg.slots, cg.epi_slots) > 4;
  // compiled programs keep every operator's values in registers: large
  // groups get the whole register file of the SM
  ge.compiled = !(o.flags & FG_FLAG_INTERPRET);
  ge.min_blocks = ge.compiled ? (cg.dag.size() + cg.epi_dag.size() <= 48 ? 2 : 1) : (ge.big ? 1 : 2);
  const int ctas = std::min(cg.ctas_per_sm, ge.min_blocks);
  ge.min_blocks = ctas;
  ge.smem = cg.smem_bytes;
  if (cg.exec == FG_EXEC_REDUCE) {
    p.red_op = cg.red_op;
    // units are (32-row strip, run of column tiles), walked in row-major
    // order
    const int unit = (o.flags >> 16) & 0xff;
    int tps, nsplit;
    if (unit > 0) {
      tps = std::min(p.ntc, unit);
    } else {
      // whole rows per unit when there is a strip for every SM (no combine
      // across CTAs: measured faster than any split there); otherwise the
      // fewest column splits per strip that spread the units evenly over the
      // SMs (an SM's share within 5 % of the busiest one's), each unit at
      // least 4 tiles long to amortise its combine step
      tps = p.ntc;
      double best = p.ntr >= nsm ? 2.0 : 0.0;
      for (int sp = 1; sp <= 64 && best < 1.5; ++sp) {
        const int t = (p.ntc + sp - 1) / sp;
        if (t < 4 && sp > 1) break;
        const int64_t units = (int64_t)p.ntr * ((p.ntc + t - 1) / t);
        const double per_sm = (double)units / nsm;
        const double balance = per_sm / std::ceil(per_sm);
        if (balance > best + 1e-9) {
          best = balance;
          tps = t;
        }
        if (balance >= 0.95) break;
      }
    }
    nsplit = (p.ntc + tps - 1) / tps;
    p.nsplit = nsplit;
    p.tiles_per_split = tps;
    p.nunits = p.ntr * nsplit;
    cg.nsplit = nsplit;
    cg.tiles_per_split = tps;
    ge.grid = std::max(1, std::min(p.nunits, ctas * nsm));
  } else {
    ge.grid = std::max(1, std::min(p.ntiles, ctas * nsm));
  }
  // The direct kernel reads the leaves straight from global memory, one warp
  // per frame row segment, without the shared-memory pipeline: for small
  // groups (rows of at most 1024 columns, so that a wide single-row frame
  // does not fall to one warp), and for row reductions of at least 8192 row
  // segments whose leaves are all read row by row (each warp's contiguous
  // run of a row keeps DRAM pages busier than the pipeline's 32-row tiles
  // do).  Compiled programs without extra outputs or shifted tuple fields
  // only; not with the failure-injection hook, whose point is the pipeline's
  // bounded waits.  Flag bit 28 turns it off.
  bool shifted = false, rowwise = true;
  for (const LeafUse& l : cg.leaves) {
    shifted |= l.map.shift != 0;
    rowwise &= l.cls == LEAF_IDENT || l.cls == LEAF_COL || l.cls == LEAF_ROW;
  }
  // warps per row: rows of 2048 columns or more split into segments of at
  // least 1024 (a warp's run of 4 KB), up to four per row (one CTA)
  p.seg = cg.exec == FG_EXEC_REDUCE ? (cg.FC >= 4096 ? 4 : cg.FC >= 2048 ? 2 : 1) : 1;
  const bool small = cg.alg_bytes <= kSmallGroupBytes && cg.FC <= 4 * 32 * 8;
  const bool rows = cg.exec == FG_EXEC_REDUCE && rowwise && cg.FR * p.seg >= kDirectMinWarps && cg.FC >= 4 * 32 * 8;
  ge.small = ge.compiled && (small || rows) && cg.xout_values.empty() && !shifted &&
             !(o.flags & FG_FLAG_INJECT_NO_LOADS) && !(o.flags & FG_FLAG_NO_SMALL);
  // A large direct launch waits for the previous kernel to end instead,
  // unless that was a direct launch too: placed early behind a pipelined
  // kernel, its CTAs land on SMs whose on-chip memory is split for that
  // kernel's shared-memory ring, and an SM that keeps taking new CTAs never
  // drains to change the split (the scaled RNNLM chain, row sum then sigmoid
  // group, launched back to back: 100 us with early launch, 85 without).
  ge.small_pdl = small;
  p.seg_cols = p.seg == 1 ? (int32_t)cg.FC : (int32_t)((cg.FC + 256 * p.seg - 1) / (256 * p.seg) * 256);
  const int64_t warps = cg.FR * p.seg;
  ge.grid_small = (int)std::max<int64_t>(1, (warps + kSmallThreads / 32 - 1) / (kSmallThreads / 32));
}

int gemm_box_bytes(int cls) {
  switch (cls) {
    case LEAF_IDENT: case LEAF_TRANS: return kGemmM * kGemmChunk * 4;
    case LEAF_COL: return kGemmChunk * 4;
    case LEAF_ROW: return kGemmM * 4;
    default: return 0;
  }
}

// Static part of the kernel parameters of a GEMM-epilogue group.
void prepare_gemm(GroupExec& ge, const BuildOpts& o, int nsm, const Graph& g) {
  CompiledGroup& cg = ge.cg;
  const int a_mn = cg.mm_ta ? 1 : 0, b_mn = cg.mm_tb ? 0 : 1;
  // TMA rows must be 16-byte multiples: the contiguous extent of each operand
  const int64_t a_inner = a_mn ? cg.M : cg.K, b_inner = b_mn ? cg.N : cg.K;
  if (a_inner % 8 || b_inner % 8)
    throw CompileError{FG_EUNSUPPORTED, "matmul operands need a contiguous extent that is a multiple of 8"};
  if (cg.N % 4) throw CompileError{FG_EUNSUPPORTED, "matmul output width must be a multiple of 4"};
  if (cg.M >= (1LL << 31) || cg.N >= (1LL << 31) || cg.K >= (1LL << 31))
    throw CompileError{FG_EUNSUPPORTED, "matmul extent too large"};
  (void)g;
  ge.mp.reset(new GemmParams());
  GemmParams& p = *ge.mp;
  std::memset(&p, 0, sizeof(p));
  if (cg.prog.size() > (size_t)kMaxProg) throw CompileError{FG_EUNSUPPORTED, "epilogue program too long"};
  std::copy(cg.prog.begin(), cg.prog.end(), p.prog);
  p.nprog = (int)cg.prog.size();
  p.nleaves = (int)cg.leaves.size();
  int mi = 0, tx = 0;
  for (size_t i = 0; i < cg.leaves.size(); ++i) {
    bool staged = cg.leaves[i].cls != LEAF_GATHER;
    fill_leaf_desc(p.leaves[i], cg.leaves[i], staged ? cg.leaf_stage_off[i] : -1, staged ? mi : -1, cg.FC);
    if (staged) {
      ++mi;
      tx += gemm_box_bytes(cg.leaves[i].cls);
    }
  }
  p.nstaged = mi;
  p.M = (int32_t)cg.M;
  p.N = (int32_t)cg.N;
  p.K = (int32_t)cg.K;
  p.ntm = (int32_t)((cg.M + kGemmM - 1) / kGemmM);
  p.ntn = (int32_t)((cg.N + kGemmN - 1) / kGemmN);
  p.ntiles = p.ntm * p.ntn;
  p.nkb = (int32_t)((cg.K + kGemmK - 1) / kGemmK);
  p.a_mn = a_mn;
  p.b_mn = b_mn;
  // one copy per operand half and ring slot through a 3-D view when the
  // contiguous extent splits into whole 64-element groups (the view would
  // otherwise wrap into the next row instead of reading zeros)
  p.a_3d = (a_mn ? cg.M : cg.K) % 64 == 0;
  p.b_3d = (b_mn ? cg.N : cg.K) % 64 == 0;
  p.wait_limit_ns = o.wait_limit_ns;
  p.epi_tx_bytes = tx;
  p.inject = (o.flags & FG_FLAG_INJECT_NO_LOADS) ? 1 : 0;
  // an IDENT leaf's chunk buffer receives the result in place, so no
  // separate output buffers are needed
  p.inplace_off = -1;
  for (size_t i = 0; i < cg.leaves.size(); ++i)
    if (cg.leaves[i].cls == LEAF_IDENT) {
      p.inplace_off = cg.leaf_stage_off[i];
      break;
    }
  // Ring granularity: a ring slot holds one or two K blocks (flag bits
  // 18-19: 1 or 2, 0 = chosen); the interpreter keeps two-block slots.  The
  // kernel always runs CTA pairs (2-CTA clusters), whose operand copies land
  // only in the CTA that issues them.
  ge.compiled = !(o.flags & FG_FLAG_INTERPRET);
  const int kbf = (o.flags >> 18) & 3, sched = (o.flags >> 20) & 3;
  const int tnf = (o.flags >> 22) & 3;
  const int KB = ge.compiled && kbf == 1 ? 1 : 2;
  constexpr int CL = kGemmCluster;
  // Pair tile width (flag bits 22-23: 0 or 1 = 256, 2 = 128, 3 = 224
  // columns; the interpreter keeps 256).  128-column tiles fill the rounds of
  // a short-K launch better, but measured slower: each tile's fixed costs and
  // the doubled A traffic outweigh it.  224-column tiles make the rounds of a
  // 4096 x 4096 output come out even (304 tiles, 4 rounds on 76 pairs, where
  // 256 leaves 28 tiles for a last round cut in two) but measured slower too
  // (K = 4096: 94.2 against 90.1 us with L2 flushed, when that last round ran
  // in column halves): the main loop is close to its operand feed, and
  // 224-column tiles load about 14 % more operand bytes per flop.
  int TN = kGemmN;
  if (ge.compiled && tnf == 2) TN = 128;
  if (ge.compiled && tnf == 3) TN = 224;
  // a 224-column tile's CTA halves start at multiples of 16 columns, not of
  // 64: an N-contiguous B is read in 2-D boxes (the 3-D view addresses whole
  // 64-column groups)
  if (TN == 224 && b_mn) p.b_3d = 0;
  p.ntn = (int32_t)((cg.N + TN - 1) / TN);
  p.ntiles = p.ntm * p.ntn;
  cg.gemm_kb = KB;
  cg.gemm_tn = TN;
  // operand ring and epilogue-leaf ring depths that fit 227 KB, in order of
  // preference: long K needs a deep operand ring (its feed is latency bound),
  // short K a deep leaf ring (the epilogue streams the leaves from HBM).  A
  // ring slot holds KB K blocks of the CTA's 128 rows of A and of its half of
  // B's columns.
  // Shared memory: alignment slack, the operand ring, the leaf stages (a
  // stage of column or row vectors alone needs 128-byte alignment, not the
  // 1024 of a swizzled box), the output staging and 512 bytes of barriers.
  int estage = cg.stage_bytes;
  {
    bool big = false;
    int end = 0;
    for (size_t i = 0; i < cg.leaves.size(); ++i)
      if (cg.leaves[i].cls != LEAF_GATHER) {
        big |= gemm_box_bytes(cg.leaves[i].cls) >= 1024;
        end = std::max(end, cg.leaf_stage_off[i] + (gemm_box_bytes(cg.leaves[i].cls) + 127) / 128 * 128);
      }
    if (!big && end > 0) estage = end;
  }
  p.epi_stage_bytes = estage;
  const int limit = 227 * 1024 - 64;   // less the kernel's static shared variables
  const int fixed = 1024 + 512 + (p.inplace_off >= 0 ? 0 : 2 * kGemmM * kGemmChunk * 4);
  auto leaf_area = [&](int n) { return (n * estage + 1023) / 1024 * 1024; };
  const int stage = KB * (kGemmM + (TN == 224 ? 128 : TN / 2)) * kGemmK * 2;   // as the kernel's kBStage
  int ns = 0, ne = 0;
  static const std::vector<std::pair<int, int>> prefs_short = {{2, 6}, {2, 5}, {2, 4}, {2, 3}, {2, 2}};
  static const std::vector<std::pair<int, int>> prefs_long = {{3, 2}, {2, 4}, {2, 3}, {2, 2}};
  const bool short_k = p.nkb <= 16 && estage > 0;
  // results written in place leave through the epilogue warps' own stores
  // (short K: the leaf stream is the whole load, and one producer thread
  // issuing a copy and waiting for its read per chunk falls behind) or
  // through the leaf producer, one copy per chunk before it reloads the
  // buffer (long K: no epilogue warp waits for a copy, which shortens the
  // exposed last epilogue); flag bits 24-25: 1 = producer, 2 = warps, 0 =
  // chosen
  {
    const int stf = (o.flags >> 24) & 3;
    p.wstore = p.inplace_off >= 0 && (stf == 2 || (stf == 0 && short_k)) ? 1 : 0;
  }
  // flag bits 29-30: the operand ring's bytes (1 = 64 KB, 2 = 96 KB, 3 =
  // 128 KB; 0 = chosen), the leaf ring taking what is left
  const int ringf = (o.flags >> 29) & 3;
  if (ringf) {
    const int qs = (ringf + 1) * 32 * 1024 / stage;
    for (int q = 8; q >= 2 && !ns; --q)
      if (qs >= 1 && fixed + qs * stage + leaf_area(q) <= limit) {
        ns = qs;
        ne = q;
      }
  }
  for (const auto& q : short_k ? prefs_short : prefs_long) {
    // the same bytes in flight with one-block slots: twice as many
    const int qs = q.first * (2 / KB);
    if (!ns && fixed + qs * stage + leaf_area(q.second) <= limit) {
      ns = qs;
      ne = q.second;
    }
  }
  if (!ns) throw CompileError{FG_EUNSUPPORTED, "GEMM epilogue stages do not fit in shared memory"};
  // the CTA's last item stages each TMEM lane quarter's results (and the
  // other piece's partial) in TN * 128 bytes of the idle operand ring, when
  // the ring holds that much
  p.last_ring = ns * stage >= 4 * TN * 128 ? 1 : 0;
  // small leaf chunks (column or row vectors): as many leaf buffers as still
  // fit, up to the barriers there are (each chunk's load is a round trip)
  while (estage > 0 && ne < 8 && fixed + ns * stage + leaf_area(ne + 1) <= limit) ++ne;
  p.nstages = ns;
  p.n_epi_bufs = ne;
  ge.smem = fixed + ns * stage + leaf_area(ne);
  // more than half of an SM's shared memory: one CTA per SM, so no two CTAs
  // ever compete for the SM's TMEM
  ge.smem = std::max(ge.smem, 120 * 1024);
  cg.nstages = ns;
  ge.big = cg.depth > 4 || cg.slots > 4;
  ge.min_blocks = 1;
  // units: the pair's 256 rows x TN columns; one CTA per SM, as many pairs
  // as run at once (flag bits 8-15, when set, cap them: a test hook for the
  // split schedules)
  const int nslots = (p.nkb + KB - 1) / KB;
  const int units = ((p.ntm + 1) / 2) * p.ntn;
  p.nunits = units;
  int avail = gemm_max_clusters(ge.smem);
  if (avail <= 0) avail = nsm / CL;
  int ncl = std::max(1, std::min(units, avail));
  const int cap = (o.flags >> 8) & 0xff;
  if (cap > 0) ncl = std::min(ncl, cap);
  ge.grid = CL * ncl;
  p.nfull = units;
  p.split = 1;
  p.sk = 0;
  p.nsplit_n = 0;
  const int tail = units % ncl;
  if (TN == 224) {
    // plain round robin: 224-column tiles are chosen for rounds that come out
    // even (the split tails' chunk bookkeeping assumes an even chunk count)
  } else if (sched == 2) {
    // every cluster takes an equal share of all units' ring slots; a share
    // spans at least one unit, so a unit is cut at most once
    if (units > ncl && tail > 0) {
      p.sk = 1;
      p.split = 2;
    }
  } else if (units > ncl && tail > 0 && 2 * tail <= ncl && TN == kGemmN &&
             (sched == 3 || (sched == 0 && p.nkb < 64))) {
    // cut the last round's units into their two column halves over the
    // pairs it would leave idle: each half runs all of K and its own
    // epilogue, with no partial sums to exchange; a half moves 3/4 of a
    // tile's operand bytes for half its flops.  Measured against symmetric
    // K pieces (below): K=1024 38.9 against 43.0 us, K=2048 53.3 against
    // 59.4 us with L2 flushed; from 64 K blocks the K pieces win (K=4096
    // 88.1-90.1 against 91.2-92.1 us flushed, 87 against 89 back to back)
    p.nfull = units - tail;
    p.split = 2;
    p.nsplit_n = 1;
    p.split_at = nslots;
  } else if (units > ncl && tail > 0 && 2 * tail <= ncl && p.nkb >= 16 && (sched == 1 || sched == 0)) {
    // split the last round's units along K into equal halves over the pairs
    // it would leave idle, when K is long enough for the halves to outweigh
    // the partial sums' traffic: both pieces run full-width MMAs, then each
    // hands the other its partial of the other's column half and finishes
    // its own half (two pieces: their sum does not depend on which ends
    // last)
    p.nfull = units - tail;
    p.split = 2;
    p.ksym = 1;
    p.split_at = std::max(1, nslots / 2);
  }
}

GroupExec make_exec(const Graph& g, const std::vector<int32_t>& nodes, const BuildOpts& o, int nsm) {
  GroupExec ge;
  try {
    ge.cg = compile_group(g, nodes);
    if (!ge.cg.xout_values.empty() && (o.flags & FG_FLAG_INTERPRET))
      throw CompileError{FG_EUNSUPPORTED, "groups with extra outputs run compiled programs only"};
    if (ge.cg.needs_jit && (o.flags & FG_FLAG_INTERPRET))
      throw CompileError{FG_EUNSUPPORTED, "groups with tuples run compiled programs only"};
    plan_staging(g, ge.cg, o);
    if (ge.cg.exec == FG_EXEC_GEMM) {
      prepare_gemm(ge, o, nsm, g);
    } else {
      prepare_group(ge, o, nsm);
    }
  } catch (const CompileError& e) {
    ge.compile_status = e.st;
    ge.compile_error = e.msg;
    ge.cg.nodes = nodes;
    std::sort(ge.cg.nodes.begin(), ge.cg.nodes.end());
    ge.cg.sink = ge.cg.nodes.back();
    ge.cg.out_value = g.nodes[ge.cg.sink].value;
  }
  return ge;
}

fg_status alloc_device(fg_plan* p, GroupExec& ge) {
  if (ge.compile_status == FG_OK && ge.mp) {
    GemmParams& mp = *ge.mp;
    mp.err = p->d_err;
    if (mp.split > 1 && !mp.nsplit_n) {
      // split units: the last round's (round robin), or one per share
      // boundary (stream-K); two pieces each
      constexpr int CL = kGemmCluster;
      const size_t keys = mp.sk ? (size_t)(ge.grid / CL - 1) : (size_t)(mp.nunits - mp.nfull);
      cudaError_t e = cudaMalloc(&ge.scratch, sizeof(float) * keys * 2 * CL * kGemmM * ge.cg.gemm_tn);
      if (e != cudaSuccess) return cuda_err(e, "cudaMalloc(split-tail workspace)");
      ge.counter_bytes = sizeof(int32_t) * keys * 2 * CL * 8;   // per piece for symmetric pieces
      e = cudaMalloc(&ge.counters, ge.counter_bytes);
      if (e != cudaSuccess) return cuda_err(e, "cudaMalloc(split-tail counters)");
      e = cudaMemset(ge.counters, 0, ge.counter_bytes);
      if (e != cudaSuccess) return cuda_err(e, "cudaMemset(split-tail counters)");
      mp.ws = ge.scratch;
      mp.ws_cnt = ge.counters;
    }
  }
  if (ge.compile_status != FG_OK || !ge.gp) return FG_OK;
  GroupParams& gp = *ge.gp;
  gp.err = p->d_err;
  if (ge.cg.exec == FG_EXEC_ELEMWISE) {
    // the claim counter of the tiles' dynamic distribution
    cudaError_t e = cudaMalloc(&ge.sched, sizeof(unsigned long long));
    if (e != cudaSuccess) return cuda_err(e, "cudaMalloc(work counter)");
    e = cudaMemset(ge.sched, 0, sizeof(unsigned long long));
    if (e != cudaSuccess) return cuda_err(e, "cudaMemset(work counter)");
    gp.sched = ge.sched;
  }
  if (ge.cg.exec == FG_EXEC_REDUCE && gp.nsplit > 1) {
    cudaError_t e = cudaMalloc(&ge.scratch, sizeof(float) * (size_t)gp.nsplit * gp.FR);
    if (e != cudaSuccess) return cuda_err(e, "cudaMalloc(reduce scratch)");
    ge.counter_bytes = sizeof(int32_t) * (size_t)gp.ntr;
    e = cudaMalloc(&ge.counters, ge.counter_bytes);
    if (e != cudaSuccess) return cuda_err(e, "cudaMalloc(reduce counters)");
    e = cudaMemset(ge.counters, 0, ge.counter_bytes);
    if (e != cudaSuccess) return cuda_err(e, "cudaMemset(reduce counters)");
    gp.scratch = ge.scratch;
    gp.counters = ge.counters;
  }
  return FG_OK;
}

void free_exec(GroupExec& ge) {
  if (ge.scratch) cudaFree(ge.scratch);
  if (ge.counters) cudaFree(ge.counters);
  if (ge.sched) cudaFree(ge.sched);
  ge.scratch = nullptr;
  ge.counters = nullptr;
  ge.sched = nullptr;
}

// ---- tensor maps -----------------------------------------------------------
fg_status encode(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
                 const uint32_t* box, bool swizzle, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32) {
  EncodeFn fn = encode_fn();
  if (!fn) return err(FG_ECUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t d[5], s[5];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
  CUresult r = fn(m, dt, rank, const_cast<void*>(ptr), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return err(FG_ECUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return FG_OK;
}

// Tensor map of a leaf (or the output, cls = LEAF_IDENT) for a frame
// [FR, FC] and a tile of TR x TC.
fg_status leaf_map(CUtensorMap* m, const void* ptr, int cls, int64_t FR, int64_t FC, int TR, int TC) {
  uint64_t dims[2], strides[1];
  uint32_t box[2];
  switch (cls) {
    case LEAF_IDENT:
      dims[0] = FC; dims[1] = FR;
      strides[0] = FR == 1 ? round_up(FC * 4, 16) : FC * 4;
      box[0] = 32; box[1] = TR;
      return encode(m, ptr, 2, dims, strides, box, true);
    case LEAF_TRANS:
      dims[0] = FR; dims[1] = FC;
      strides[0] = FC == 1 ? round_up(FR * 4, 16) : FR * 4;
      box[0] = 32; box[1] = TC;
      return encode(m, ptr, 2, dims, strides, box, true);
    case LEAF_COL:
      dims[0] = FC; box[0] = TC;
      return encode(m, ptr, 1, dims, strides, box, false);
    case LEAF_ROW:
      dims[0] = FR; box[0] = TR;
      return encode(m, ptr, 1, dims, strides, box, false);
    default:
      return err(FG_EINVAL, "internal: map for a gathered leaf");
  }
}

fg_status check_ptr(const void* p, int32_t vid) {
  if (!p) return err(FG_EINVAL, "null device pointer for value " + std::to_string(vid));
  if (reinterpret_cast<uintptr_t>(p) % 16) return err(FG_EINVAL, "value " + std::to_string(vid) + " is not 16-byte aligned");
  return FG_OK;
}

fg_status launch_gemm(GroupExec& ge, void* const* ptrs, void* stream) {
  const CompiledGroup& cg = ge.cg;
  GemmParams& gp = *ge.mp;
  std::vector<const void*> key{ptrs[cg.mm_a], ptrs[cg.mm_b], ptrs[cg.out_value]};
  for (int32_t v : cg.leaf_values) key.push_back(ptrs[v]);
  if (key != ge.last_ptrs) {
    for (int32_t v : cg.leaf_values) if (fg_status st = check_ptr(ptrs[v], v)) return st;
    if (fg_status st = check_ptr(ptrs[cg.out_value], cg.out_value)) return st;
    {
      // A: [K, M] (M contiguous) when transposed, else [M, K]
      // 3-D views (one copy per operand half and ring slot):
      //   MN-major [extent/64][K][64], box 64 x 128 K rows x 2 groups;
      //   K-major  [K/64][rows][64],   box 64 x 128 rows x 2 K blocks.
      // Otherwise 2-D boxes: MN-major 64 x 64, K-major 64 x 128 rows.
      // With KB K blocks per ring slot the 3-D boxes cover KB * 64 K rows
      // (MN-major) or KB K blocks (K-major), over a half's R rows (A: 128;
      // B: half the tile's columns).
      uint64_t dims[3], strides[2];
      uint32_t box[3];
      const int KB = cg.gemm_kb;
      auto view = [&](bool mn, bool v3, int64_t rows, int R) {
        const int64_t inner = mn ? rows : cg.K, outer = mn ? cg.K : rows;
        if (v3) {
          dims[0] = 64; dims[1] = outer; dims[2] = inner / 64; strides[0] = inner * 2; strides[1] = 128;
          box[0] = 64; box[1] = mn ? 64 * KB : R; box[2] = mn ? R / 64 : KB;
          return 3;
        }
        dims[0] = inner; dims[1] = outer; strides[0] = inner * 2; box[0] = 64;
        box[1] = mn ? 64 : R;
        return 2;
      };
      int rank = view(gp.a_mn, gp.a_3d, cg.M, kGemmM);
      if (fg_status st = encode(&gp.mapA, ptrs[cg.mm_a], rank, dims, strides, box, true,
                                CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
        return st;
      // B: [K, N] (N contiguous), or [N, K] when transposed; each CTA of a
      // pair stages its half of the tile's columns
      rank = view(gp.b_mn, gp.b_3d, cg.N, cg.gemm_tn == 224 ? 128 : cg.gemm_tn / 2);
      if (fg_status st = encode(&gp.mapB, ptrs[cg.mm_b], rank, dims, strides, box, true,
                                CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
        return st;
      if (gp.nsplit_n) {
        // a unit's column half: each CTA stages a quarter of the tile's columns
        rank = view(gp.b_mn, gp.b_3d, cg.N, cg.gemm_tn / 4);
        if (fg_status st = encode(&gp.mapB2, ptrs[cg.mm_b], rank, dims, strides, box, true,
                                  CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
          return st;
      }
    }
    for (size_t i = 0; i < cg.leaves.size(); ++i) {
      const LeafUse& l = cg.leaves[i];
      LeafDesc& d = gp.leaves[i];
      d.ptr = static_cast<const float*>(ptrs[l.value]);
      if (l.cls != LEAF_GATHER)
        if (fg_status st = leaf_map(&gp.maps[d.map_idx], ptrs[l.value], l.cls, cg.FR, cg.FC, kGemmM, kGemmChunk))
          return st;
    }
    gp.out = static_cast<float*>(ptrs[cg.out_value]);
    // each epilogue warp stores its own 32 x 32 box; results written in
    // place leave a whole 128 x 32 chunk at a time
    if (fg_status st = leaf_map(&gp.maps[kMaxStaged], ptrs[cg.out_value], LEAF_IDENT, cg.FR, cg.FC, 32, kGemmChunk))
      return st;
    if (fg_status st = leaf_map(&gp.maps[kMaxStaged + 1], ptrs[cg.out_value], LEAF_IDENT, cg.FR, cg.FC, kGemmM, kGemmChunk))
      return st;
    ge.last_ptrs = key;
  }
  cudaError_t e = ge.fn ? jit_launch_gemm(ge.fn, gp, ge.grid, ge.smem, static_cast<cudaStream_t>(stream))
                        : launch_gemm_kernel(gp, ge.big ? 1 : 0, ge.grid, ge.smem, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    ge.last_ptrs.clear();
    return cuda_err(e, "GEMM kernel launch");
  }
  return FG_OK;
}

// Whether the last kernel this library launched on a stream was the direct
// kernel; returns that and records the new launch's kind.  A large direct
// launch starts early only behind another direct launch (any other of this
// library's kernels uses a shared-memory ring).  Only speed depends on it:
// a kernel launched early waits for its predecessor all the same.
bool swap_last_direct(void* stream, bool direct) {
  static std::mutex mu;
  static std::unordered_map<void*, bool> last;
  std::lock_guard<std::mutex> g(mu);
  // bounded: forgetting the streams costs at most one early start each
  if (last.size() >= 1024 && !last.count(stream)) last.clear();
  bool& v = last[stream];
  const bool prev = v;
  v = direct;
  return prev;
}

fg_status launch_exec(fg_plan* p, GroupExec& ge, void* const* ptrs, void* stream) {
  if (ge.compile_status != FG_OK) return err(ge.compile_status, ge.compile_error);
  if (!p->has_device) return err(FG_ECUDA, "no CUDA device: the plan is host-only");
  if (!ptrs) return err(FG_EINVAL, "null value_ptrs");
  if (ge.cg.exec == FG_EXEC_GEMM) {
    if (!ptrs[ge.cg.mm_a] || !ptrs[ge.cg.mm_b]) return err(FG_EINVAL, "null matmul operand");
    if (reinterpret_cast<uintptr_t>(ptrs[ge.cg.mm_a]) % 16 || reinterpret_cast<uintptr_t>(ptrs[ge.cg.mm_b]) % 16)
      return err(FG_EINVAL, "matmul operands must be 16-byte aligned");
    swap_last_direct(stream, false);
    return launch_gemm(ge, ptrs, stream);
  }
  const CompiledGroup& cg = ge.cg;
  GroupParams& gp = *ge.gp;
  // cache key: the pointers this group reads and writes
  std::vector<const void*> key;
  for (int32_t v : cg.leaf_values) key.push_back(ptrs[v]);
  for (int32_t v : cg.epi_leaf_values) key.push_back(ptrs[v]);
  key.push_back(ptrs[cg.out_value]);
  for (int32_t v : cg.xout_values) key.push_back(ptrs[v]);
  if (key != ge.last_ptrs) {
    for (int32_t v : cg.xout_values) if (fg_status st = check_ptr(ptrs[v], v)) return st;
    for (size_t j = 0; j < cg.xout_values.size(); ++j) gp.xout[j].ptr = static_cast<float*>(ptrs[cg.xout_values[j]]);
    for (int32_t v : cg.leaf_values) if (fg_status st = check_ptr(ptrs[v], v)) return st;
    for (int32_t v : cg.epi_leaf_values) if (fg_status st = check_ptr(ptrs[v], v)) return st;
    if (fg_status st = check_ptr(ptrs[cg.out_value], cg.out_value)) return st;
    for (size_t i = 0; i < cg.leaves.size(); ++i) {
      const LeafUse& l = cg.leaves[i];
      LeafDesc& d = gp.leaves[i];
      d.ptr = static_cast<const float*>(ptrs[l.value]);
      if (l.cls != LEAF_GATHER)
        if (fg_status st = leaf_map(&gp.maps[d.map_idx], ptrs[l.value], l.cls, cg.FR, cg.FC, kTileR, kTileC)) return st;
    }
    for (size_t i = 0; i < cg.epi_leaf_values.size(); ++i)
      gp.epi_leaf[i] = static_cast<const float*>(ptrs[cg.epi_leaf_values[i]]);
    gp.out = static_cast<float*>(ptrs[cg.out_value]);
    if (cg.exec == FG_EXEC_ELEMWISE && cg.out_tma == 1)
      if (fg_status st = leaf_map(&gp.maps[kMaxStaged], ptrs[cg.out_value], LEAF_IDENT, cg.FR, cg.FC, kTileR, kTileC))
        return st;
    if (cg.xout_tma)
      for (size_t j = 0; j < cg.xout_values.size(); ++j) {
        // a warp's slice: 32 frame rows x 8 frame columns, or its transpose
        const bool id = cg.xout_cls[j] == LEAF_IDENT;
        uint64_t dims[2] = {(uint64_t)(id ? cg.FC : cg.FR), (uint64_t)(id ? cg.FR : cg.FC)};
        const int64_t inner = id ? cg.FC : cg.FR, outer = id ? cg.FR : cg.FC;
        uint64_t strides[1] = {(uint64_t)(outer == 1 ? round_up(inner * 4, 16) : inner * 4)};
        uint32_t box[2] = {id ? 8u : (uint32_t)kTileR, id ? (uint32_t)kTileR : 8u};
        if (fg_status st = encode(&gp.xmaps[j], ptrs[cg.xout_values[j]], 2, dims, strides, box, false)) return st;
      }
    if (cg.exec == FG_EXEC_ELEMWISE && cg.out_tma == 2) {
      // one warp's 32 x 8 slice per store
      uint64_t dims[2] = {(uint64_t)cg.FC, (uint64_t)cg.FR};
      uint64_t strides[1] = {(uint64_t)(cg.FR == 1 ? round_up(cg.FC * 4, 16) : cg.FC * 4)};
      uint32_t box[2] = {8, (uint32_t)kTileR};
      if (fg_status st = encode(&gp.maps[kMaxStaged], ptrs[cg.out_value], 2, dims, strides, box, false)) return st;
    }
    ge.last_ptrs = key;
  }
  const bool direct = ge.small && ge.fn_small;
  const bool after_direct = swap_last_direct(stream, direct);
  cudaError_t e = direct
                      ? jit_launch_any(ge.fn_small, &gp, ge.grid_small, kSmallThreads,
                                       gp.seg > 1 ? kSmallThreads / 32 * (int)sizeof(float) : 0,
                                       static_cast<cudaStream_t>(stream),
                                       ge.small_pdl || after_direct)
                  : ge.fn ? jit_launch(ge.fn, gp, ge.grid, ge.smem, static_cast<cudaStream_t>(stream))
                        : launch_group_kernel(gp, cg.exec == FG_EXEC_REDUCE ? 1 : 0, ge.big ? 1 : 0, ge.grid,
                                              ge.smem, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    ge.last_ptrs.clear();
    return cuda_err(e, "group kernel launch");
  }
  return FG_OK;
}

fg_status build_opts_from(const fg_build_opts* opts, BuildOpts& b) {
  fg_build_opts o;
  fg_build_opts_default(&o);
  if (opts) o = *opts;
  if (o.max_fused_ops < 1 || o.max_args < 2) return err(FG_EINVAL, "max_fused_ops >= 1 and max_args >= 2 required");
  b.max_fused_ops = o.max_fused_ops;
  b.max_args = o.max_args;
  b.allow_reduce_epilogue = o.allow_reduce_epilogue;
  b.wait_limit_ns = o.wait_limit_ns > 0 ? o.wait_limit_ns : 2000000000LL;
  b.flags = o.flags;
  return FG_OK;
}

// A plan for the given groups (in launch order): compiled programs, device
// tables and the unfused single-operator programs.
fg_status build_plan(const Graph& g, const BuildOpts& o, const std::vector<std::vector<int32_t>>& groups,
                     const std::vector<int32_t>& group_of, const std::vector<int32_t>& ipdom, fg_plan** out) {
  std::unique_ptr<fg_plan> p(new (std::nothrow) fg_plan());
  if (!p) return err(FG_ENOMEM, "out of host memory");
  p->g = g;
  p->opts = o;
  p->group_of = group_of;
  p->ipdom = ipdom;
  p->has_device = device_present(&p->nsm);
  for (const auto& nodes : groups) p->groups.push_back(make_exec(p->g, nodes, p->opts, p->nsm));
  for (size_t i = 0; i < p->g.nodes.size(); ++i)
    p->singles.push_back(make_exec(p->g, {(int32_t)i}, p->opts, p->nsm));
  if (p->has_device) {
    cudaError_t e = cudaMalloc(&p->d_err, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_err(e, "cudaMalloc(error flag)");
    e = cudaMemset(p->d_err, 0, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_err(e, "cudaMemset(error flag)");
    for (auto& ge : p->groups) if (fg_status st = alloc_device(p.get(), ge)) return st;
    for (auto& ge : p->singles) if (fg_status st = alloc_device(p.get(), ge)) return st;
    // compile every group program (and every single-operator program) once
    std::vector<GroupExec*> todo;
    std::vector<std::string> srcs;
    for (auto* v : {&p->groups, &p->singles})
      for (auto& ge : *v)
        if (ge.compile_status == FG_OK && (ge.gp || ge.mp) && ge.compiled) {
          todo.push_back(&ge);
          srcs.push_back(jit_source(ge.cg, ge.min_blocks, ge.small ? ge.gp->seg : 0));
        }
    if (!todo.empty()) {
      std::vector<void*> fns, smalls;
      std::string msg = jit_compile(srcs, fns, &smalls);
      if (!msg.empty()) return err(FG_ECUDA, msg);
      for (size_t i = 0; i < todo.size(); ++i) {
        todo[i]->fn = fns[i];
        todo[i]->fn_small = smalls[i];
      }
    }
  }
  *out = p.release();
  return FG_OK;
}

}  // namespace

extern "C" {

fg_status fg_build_groups(const fg_graph* gh, const fg_build_opts* opts, fg_plan** out) {
  if (!gh || !out) return err(FG_EINVAL, "null argument");
  *out = nullptr;
  BuildOpts o;
  if (fg_status st = build_opts_from(opts, o)) return st;
  if (gh->g.nodes.empty()) return err(FG_EINVAL, "graph has no operators");
  std::vector<int32_t> group_of, ipdom;
  partition(gh->g, o, group_of, ipdom);
  std::vector<std::vector<int32_t>> groups;
  for (size_t s = 0; s < group_of.size(); ++s)
    if (group_of[s] == (int32_t)s) {
      groups.emplace_back();
      for (size_t i = 0; i < group_of.size(); ++i)
        if (group_of[i] == (int32_t)s) groups.back().push_back((int32_t)i);
    }
  return build_plan(gh->g, o, groups, group_of, ipdom, out);
}

// ---- explicit fusion ---------------------------------------------------------
fg_status fg_partition_create(const fg_graph* gh, const fg_build_opts* opts, int32_t from_fuseops,
                              fg_partition** out) {
  if (!gh || !out) return err(FG_EINVAL, "null argument");
  *out = nullptr;
  BuildOpts o;
  if (fg_status st = build_opts_from(opts, o)) return st;
  if (gh->g.nodes.empty()) return err(FG_EINVAL, "graph has no operators");
  std::unique_ptr<fg_partition> p(new (std::nothrow) fg_partition());
  if (!p) return err(FG_ENOMEM, "out of host memory");
  p->opts = o;
  p->P = singleton_partition(gh->g, o);
  if (from_fuseops) {
    std::vector<int32_t> group_of, ipdom;
    partition(gh->g, o, group_of, ipdom);
    // label = the group's smallest node id
    std::vector<int32_t> first(group_of.size(), -1);
    for (size_t i = 0; i < group_of.size(); ++i)
      if (first[group_of[i]] < 0) first[group_of[i]] = (int32_t)i;
    for (size_t i = 0; i < group_of.size(); ++i) p->P.label[i] = first[group_of[i]];
  }
  *out = p.release();
  return FG_OK;
}

namespace {
// A fused group must run as one kernel within the build options' bounds.
GroupCheck executable(const BuildOpts& o) {
  return [o](const Graph& g, const std::vector<int32_t>& nodes) {
    // an opaque operator stays alone (TVM "Operator Fusion", Operator Pattern
    // Classification: opaque operators are not fused)
    if (nodes.size() > 1)
      for (int32_t x : nodes)
        if (op_kind(g.nodes[x].op) == K_OPAQUE) throw CompileError{FG_EUNSUPPORTED, "an opaque operator stays alone"};
    GroupExec ge = make_exec(g, nodes, o, 148);
    if (ge.compile_status != FG_OK) throw CompileError{ge.compile_status, ge.compile_error};
    const int args = (int)(ge.cg.leaf_values.size() + ge.cg.epi_leaf_values.size() + 1 + ge.cg.xout_values.size());
    if (args > o.max_args) throw CompileError{FG_EUNSUPPORTED, "the fused group exceeds max_args"};
    if ((int)nodes.size() > o.max_fused_ops) throw CompileError{FG_EUNSUPPORTED, "the fused group exceeds max_fused_ops"};
  };
}
}  // namespace

fg_status fg_partition_fuse(fg_partition* p, int32_t node, int32_t pred, int32_t duplicate) {
  if (!p) return err(FG_EINVAL, "null partition");
  try {
    fuse_move(p->P, node, pred, duplicate != 0, executable(p->opts));
  } catch (const CompileError& e) {
    return err(e.st, e.msg);
  }
  return FG_OK;
}

fg_status fg_partition_from_patterns(const fg_graph* gh, const fg_build_opts* opts, int32_t n_patterns,
                                     const fg_pattern* patterns, fg_partition** out, int32_t* match_of) {
  if (!gh || !out || (n_patterns > 0 && !patterns) || n_patterns < 0) return err(FG_EINVAL, "null argument");
  *out = nullptr;
  BuildOpts o;
  if (fg_status st = build_opts_from(opts, o)) return st;
  if (gh->g.nodes.empty()) return err(FG_EINVAL, "graph has no operators");
  std::vector<ChainPattern> pats(n_patterns);
  for (int k = 0; k < n_patterns; ++k) {
    if (patterns[k].n_ops < 1 || !patterns[k].opcodes) return err(FG_EINVAL, "a pattern needs at least one operator");
    pats[k].ops.assign(patterns[k].opcodes, patterns[k].opcodes + patterns[k].n_ops);
    pats[k].private_intermediates = patterns[k].private_intermediates != 0;
  }
  std::unique_ptr<fg_partition> p(new (std::nothrow) fg_partition());
  if (!p) return err(FG_ENOMEM, "out of host memory");
  p->opts = o;
  std::vector<int32_t> mo;
  p->P = pattern_partition(gh->g, o, pats, executable(o), mo);
  if (match_of) std::copy(mo.begin(), mo.end(), match_of);
  *out = p.release();
  return FG_OK;
}

fg_status fg_partition_query(const fg_partition* p, int32_t* n_nodes, int32_t* group_of, int32_t* clone_of) {
  if (!p) return err(FG_EINVAL, "null partition");
  if (n_nodes) *n_nodes = (int32_t)p->P.label.size();
  if (group_of) std::copy(p->P.label.begin(), p->P.label.end(), group_of);
  if (clone_of) std::copy(p->P.clone_of.begin(), p->P.clone_of.end(), clone_of);
  return FG_OK;
}

fg_status fg_build_from_partition(const fg_partition* p, fg_plan** out) {
  if (!p || !out) return err(FG_EINVAL, "null argument");
  *out = nullptr;
  std::vector<std::vector<int32_t>> groups;
  try {
    groups = partition_groups(p->P);
  } catch (const CompileError& e) {
    return err(e.st, e.msg);
  }
  std::vector<int32_t> ipdom(p->P.label.size(), -1);
  return build_plan(p->P.g, p->opts, groups, p->P.label, ipdom, out);
}

void fg_partition_destroy(fg_partition* p) { delete p; }

void fg_plan_destroy(fg_plan* p) {
  if (!p) return;
  for (auto& ge : p->groups) free_exec(ge);
  for (auto& ge : p->singles) free_exec(ge);
  if (p->d_err) cudaFree(p->d_err);
  delete p;
}

fg_status fg_plan_query(const fg_plan* p, int32_t* n_nodes, int32_t* n_groups, int32_t* group_of, int32_t* ipdom) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (n_nodes) *n_nodes = (int32_t)p->group_of.size();
  if (n_groups) *n_groups = (int32_t)p->groups.size();
  if (group_of) std::copy(p->group_of.begin(), p->group_of.end(), group_of);
  if (ipdom) std::copy(p->ipdom.begin(), p->ipdom.end(), ipdom);
  return FG_OK;
}

fg_status fg_plan_group_info(const fg_plan* p, int32_t gid, int32_t* n_nodes, int32_t* nodes, int32_t* n_leaves,
                             int32_t* leaves, int32_t* out_value, int32_t* kind, int64_t* alg_bytes,
                             int64_t* alg_flops) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (gid < 0 || gid >= (int32_t)p->groups.size()) return err(FG_EINVAL, "unknown group id");
  const GroupExec& ge = p->groups[gid];
  const CompiledGroup& cg = ge.cg;
  if (n_nodes) *n_nodes = (int32_t)cg.nodes.size();
  if (nodes) std::copy(cg.nodes.begin(), cg.nodes.end(), nodes);
  if (n_leaves) *n_leaves = (int32_t)cg.leaf_values.size();
  if (leaves) std::copy(cg.leaf_values.begin(), cg.leaf_values.end(), leaves);
  if (out_value) *out_value = cg.out_value;
  if (kind) *kind = cg.exec;
  if (alg_bytes) *alg_bytes = cg.alg_bytes;
  if (alg_flops) *alg_flops = cg.alg_flops;
  if (ge.compile_status != FG_OK) return err(ge.compile_status, ge.compile_error);
  return FG_OK;
}

fg_status fg_plan_group_outputs(const fg_plan* p, int32_t gid, int32_t* n_out, int32_t* out_values) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (gid < 0 || gid >= (int32_t)p->groups.size()) return err(FG_EINVAL, "unknown group id");
  const CompiledGroup& cg = p->groups[gid].cg;
  if (n_out) *n_out = (int32_t)(1 + cg.xout_values.size());
  if (out_values) {
    out_values[0] = cg.out_value;
    std::copy(cg.xout_values.begin(), cg.xout_values.end(), out_values + 1);
  }
  return FG_OK;
}

fg_status fg_plan_group_exec_info(const fg_plan* p, int32_t gid, int32_t* tile_rows, int32_t* tile_cols,
                                  int32_t* stages, int32_t* n_staged, int32_t* n_gathered, int32_t* prog_len) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (gid < 0 || gid >= (int32_t)p->groups.size()) return err(FG_EINVAL, "unknown group id");
  const CompiledGroup& cg = p->groups[gid].cg;
  bool gemm = cg.exec == FG_EXEC_GEMM;
  if (tile_rows) *tile_rows = gemm ? 128 : kTileR;
  if (tile_cols) *tile_cols = gemm ? 256 : kTileC;
  if (stages) *stages = cg.nstages;
  if (n_staged) *n_staged = cg.nstaged;
  if (n_gathered) *n_gathered = cg.ngathered;
  if (prog_len) *prog_len = (int32_t)cg.prog.size();
  return FG_OK;
}

fg_status fg_plan_group_direct_info(const fg_plan* p, int32_t gid, int32_t* direct, int32_t* segments,
                                    int32_t* early_launch) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (gid < 0 || gid >= (int32_t)p->groups.size()) return err(FG_EINVAL, "unknown group id");
  const GroupExec& ge = p->groups[gid];
  const bool d = ge.small && ge.gp;
  if (direct) *direct = d ? 1 : 0;
  if (segments) *segments = d ? ge.gp->seg : 1;
  if (early_launch) *early_launch = d ? (ge.small_pdl ? 1 : 0) : 1;
  return FG_OK;
}

fg_status fg_plan_group_source(const fg_plan* p, int32_t gid, char* buf, int64_t cap, int64_t* len_out) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (gid < 0 || gid >= (int32_t)p->groups.size()) return err(FG_EINVAL, "unknown group id");
  const GroupExec& ge = p->groups[gid];
  if (ge.compile_status != FG_OK) return err(ge.compile_status, ge.compile_error);
  if (!ge.gp && !ge.mp) return err(FG_EUNSUPPORTED, "no compiled program for this group kind");
  const std::string src = jit_source(ge.cg, ge.min_blocks, ge.small && ge.gp ? ge.gp->seg : 0);
  if (len_out) *len_out = (int64_t)src.size();
  if (buf && cap > 0) {
    const size_t n = std::min<size_t>(src.size(), (size_t)cap - 1);
    std::memcpy(buf, src.data(), n);
    buf[n] = 0;
  }
  return FG_OK;
}

fg_status fg_launch_group(fg_plan* p, int32_t gid, void* const* value_ptrs, void* stream) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (gid < 0 || gid >= (int32_t)p->groups.size()) return err(FG_EINVAL, "unknown group id");
  return launch_exec(p, p->groups[gid], value_ptrs, stream);
}

fg_status fg_launch_unfused(fg_plan* p, int32_t node, void* const* value_ptrs, void* stream) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (node < 0 || node >= (int32_t)p->singles.size()) return err(FG_EINVAL, "unknown node id");
  return launch_exec(p, p->singles[node], value_ptrs, stream);
}

fg_status fg_sync_status(fg_plan* p, void* stream) {
  if (!p) return err(FG_EINVAL, "null plan");
  if (!p->has_device) return err(FG_ECUDA, "no CUDA device: the plan is host-only");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize");
  int32_t flag = 0;
  e = cudaMemcpy(&flag, p->d_err, sizeof(flag), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_err(e, "reading the device error flag");
  if (flag == 0) return FG_OK;
  cudaMemset(p->d_err, 0, sizeof(int32_t));
  // a kernel that gave up may have left split arrival counters mid-count and
  // its claim counter off the launches' count
  for (auto* v : {&p->groups, &p->singles})
    for (auto& ge : *v) {
      if (ge.counters) cudaMemset(ge.counters, 0, ge.counter_bytes);
      if (ge.sched) cudaMemset(ge.sched, 0, sizeof(unsigned long long));
    }
  if (flag == DEVERR_TIMEOUT) return err(FG_ETIMEOUT, "a device-side wait exceeded wait_limit_ns");
  return err(FG_EDEVICE, "device error flag " + std::to_string(flag));
}

// ---------------------------------------------------------------------------
// tensor fusion
fg_status tf_layout_offsets(int32_t n, const int64_t* numel, fg_dtype buf_dtype, int64_t align,
                            int64_t* offsets_out, int64_t* total_out) {
  if (n > 0 && !numel) return err(FG_EINVAL, "null argument");
  if (n <= 0) return err(FG_EINVAL, "no tensors");
  if (buf_dtype != FG_BF16 && buf_dtype != FG_F32) return err(FG_EINVAL, "unknown buffer dtype");
  if (align < 16 || (align & (align - 1))) return err(FG_EINVAL, "align_bytes must be a power of two >= 16");
  const int64_t eb = buf_dtype == FG_BF16 ? 2 : 4;
  int64_t cur = 0;
  for (int i = 0; i < n; ++i) {
    if (numel[i] < 0) return err(FG_ESHAPE, "negative element count");
    if (offsets_out) offsets_out[i] = cur;
    cur = round_up(cur + numel[i] * eb, align);
  }
  if (total_out) *total_out = cur;
  return FG_OK;
}

fg_status tf_layout_create(int32_t n, const int64_t* numel, float* const* grads, fg_dtype buf_dtype,
                           int64_t align, tf_layout** out, int64_t* offsets_out, int64_t* total_out) {
  if (!out || (n > 0 && (!numel || !grads))) return err(FG_EINVAL, "null argument");
  *out = nullptr;
  if (n <= 0) return err(FG_EINVAL, "no tensors");
  if (buf_dtype != FG_BF16 && buf_dtype != FG_F32) return err(FG_EINVAL, "unknown buffer dtype");
  if (align < 16 || (align & (align - 1))) return err(FG_EINVAL, "align_bytes must be a power of two >= 16");
  std::unique_ptr<tf_layout> l(new (std::nothrow) tf_layout());
  if (!l) return err(FG_ENOMEM, "out of host memory");
  l->n = n;
  l->buf_bf16 = buf_dtype == FG_BF16;
  const int64_t eb = l->buf_bf16 ? 2 : 4;
  int64_t cur = 0;
  for (int i = 0; i < n; ++i) {
    if (numel[i] < 0) return err(FG_ESHAPE, "negative element count");
    if (numel[i] > 0) if (fg_status st = check_ptr(grads[i], i)) return st;
    l->numel.push_back(numel[i]);
    l->grads.push_back(grads[i]);
    l->offsets.push_back(cur);
    cur = round_up(cur + numel[i] * eb, align);
  }
  l->total = cur;
  std::vector<TfChunk> ch;
  for (int i = 0; i < n; ++i) {
    l->chunk_begin.push_back((int32_t)ch.size());
    const int64_t end_bytes = l->offsets[i] + numel[i] * eb;
    const int64_t next = i + 1 < n ? l->offsets[i + 1] : l->total;
    int64_t s = 0;
    do {
      TfChunk c;
      c.tensor = grads[i];
      c.start = s;
      c.count = (int32_t)std::min<int64_t>(kTfChunk, numel[i] - s);
      c.buf_off = l->offsets[i] + s * eb;
      s += c.count;
      c.pad_bytes = s >= numel[i] ? (int32_t)(next - end_bytes) : 0;
      ch.push_back(c);
    } while (s < numel[i]);
  }
  l->nchunks = (int)ch.size();
  l->chunk_begin.push_back(l->nchunks);
  if (!device_present(nullptr)) return err(FG_ECUDA, "no CUDA device");
  const size_t table = round_up((int64_t)(sizeof(TfChunk) * ch.size()), 256);
  cudaError_t e = cudaMalloc(&l->d_chunks, table + 256);
  if (e != cudaSuccess) return cuda_err(e, "cudaMalloc(chunk table)");
  l->d_err = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(l->d_chunks) + table);
  l->d_claim = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(l->d_chunks) + table + 64);
  e = cudaMemcpy(l->d_chunks, ch.data(), sizeof(TfChunk) * ch.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(l->d_err, 0, 256);   // the error word and the claim counters
  if (e != cudaSuccess) {
    cudaFree(l->d_chunks);
    return cuda_err(e, "cudaMemcpy(chunk table)");
  }
  if (offsets_out) std::copy(l->offsets.begin(), l->offsets.end(), offsets_out);
  if (total_out) *total_out = l->total;
  *out = l.release();
  return FG_OK;
}

// Chunks [c0, c1) of the layout's table: tensors first .. first+count-1.
static fg_status tf_chunk_range(const tf_layout* l, int32_t first, int32_t count, int* c0, int* c1) {
  if (first < 0 || count < 0 || first > l->n || count > l->n - first) return err(FG_EINVAL, "tensor range out of bounds");
  *c0 = l->chunk_begin[first];
  *c1 = l->chunk_begin[first + count];
  return FG_OK;
}

fg_status tf_pack_range(const tf_layout* l, int32_t first, int32_t count, float scale, void* buf, void* stream) {
  if (!l || !buf) return err(FG_EINVAL, "null argument");
  if (reinterpret_cast<uintptr_t>(buf) % 256) return err(FG_EINVAL, "fusion buffer must be 256-byte aligned");
  int c0, c1;
  if (fg_status st = tf_chunk_range(l, first, count, &c0, &c1)) return st;
  if (c1 == c0) return FG_OK;
  int nsm = 148;
  device_present(&nsm);
  // launches over the whole layout claim their chunks dynamically
  const bool all = c0 == 0 && c1 == l->nchunks;
  swap_last_direct(stream, false);
  cudaError_t e = launch_tf_pack(l->d_chunks + c0, c1 - c0, l->buf_bf16, scale, buf,
                                 std::min(c1 - c0, tf_pack_resident(nsm)),
                                 static_cast<cudaStream_t>(stream), TfBuckets(), all ? l->d_claim : nullptr);
  return e == cudaSuccess ? FG_OK : cuda_err(e, "tf_pack launch");
}

fg_status tf_unpack_range(const tf_layout* l, int32_t first, int32_t count, float uscale, const void* buf,
                          void* stream) {
  if (!l || !buf) return err(FG_EINVAL, "null argument");
  if (reinterpret_cast<uintptr_t>(buf) % 256) return err(FG_EINVAL, "fusion buffer must be 256-byte aligned");
  int c0, c1;
  if (fg_status st = tf_chunk_range(l, first, count, &c0, &c1)) return st;
  if (c1 == c0) return FG_OK;
  int nsm = 148;
  device_present(&nsm);
  swap_last_direct(stream, false);
  cudaError_t e = launch_tf_unpack(l->d_chunks + c0, c1 - c0, l->buf_bf16, uscale, buf, std::min(c1 - c0, nsm),
                                   l->d_err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FG_OK : cuda_err(e, "tf_unpack launch");
}

fg_status tf_pack(const tf_layout* l, float scale, void* buf, void* stream) {
  if (!l) return err(FG_EINVAL, "null argument");
  return tf_pack_range(l, 0, l->n, scale, buf, stream);
}

fg_status tf_layout_set_buckets(tf_layout* l, int32_t nb, const int32_t* bounds) {
  if (!l || !bounds) return err(FG_EINVAL, "null argument");
  if (nb <= 0 || bounds[0] != 0 || bounds[nb] != l->n) return err(FG_EINVAL, "bucket bounds must run from 0 to n");
  for (int32_t b = 0; b < nb; ++b)
    if (bounds[b + 1] <= bounds[b]) return err(FG_EINVAL, "bucket bounds must increase strictly");
  // chunk -> bucket, then chunks per bucket; counts zero
  std::vector<int32_t> host((size_t)l->nchunks + 2 * (size_t)nb, 0);
  std::vector<uint32_t> per(nb);
  for (int32_t b = 0; b < nb; ++b) {
    const int c0 = l->chunk_begin[bounds[b]], c1 = l->chunk_begin[bounds[b + 1]];
    for (int c = c0; c < c1; ++c) host[c] = b;
    host[(size_t)l->nchunks + b] = c1 - c0;
    per[b] = (uint32_t)(c1 - c0);
  }
  int32_t* d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(int32_t) * host.size());
  if (e != cudaSuccess) return cuda_err(e, "cudaMalloc(bucket table)");
  e = cudaMemcpy(d, host.data(), sizeof(int32_t) * host.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(d);
    return cuda_err(e, "cudaMemcpy(bucket table)");
  }
  if (l->d_bucket) {
    // an earlier table may still be read by a pack or a stream wait in
    // flight: it is freed once the events recorded after them have completed
    l->retired.push_back(tf_layout::Retired{l->d_bucket, std::move(l->users)});
    l->users.clear();
  }
  free_retired(l, false);
  l->d_bucket = d;
  l->nb = nb;
  l->seq = 0;
  l->bucket_chunks = std::move(per);
  return FG_OK;
}

namespace {
fg_status pack_buckets(tf_layout* l, float scale, void* buf, void* stream, uint64_t* times, uint32_t seq_offset,
                       int64_t limit_ns) {
  if (!l || !buf) return err(FG_EINVAL, "null argument");
  if (!l->nb) return err(FG_EINVAL, "no bucket table (tf_layout_set_buckets)");
  if (reinterpret_cast<uintptr_t>(buf) % 256) return err(FG_EINVAL, "fusion buffer must be 256-byte aligned");
  int nsm = 148;
  device_present(&nsm);
  TfBuckets bk;
  bk.chunk_bucket = l->d_bucket;
  bk.nchunks = l->d_bucket + l->nchunks;
  bk.count = reinterpret_cast<uint32_t*>(l->d_bucket + l->nchunks + l->nb);
  bk.seq = l->seq + 1;
  // every CTA resident at once, the observer's included
  const int resident = tf_pack_resident(nsm);
  int grid = std::min(l->nchunks, std::max(1, resident - (times ? 1 : 0)));
  if (times) {
    // one more CTA, the observer
    bk.observe = reinterpret_cast<unsigned long long*>(times);
    bk.nb = l->nb;
    bk.seq_offset = seq_offset;
    bk.limit_ns = limit_ns;
    bk.err = l->d_err;
    grid += 1;
  }
  swap_last_direct(stream, false);
  cudaError_t e = launch_tf_pack(l->d_chunks, l->nchunks, l->buf_bf16, scale, buf, grid,
                                 static_cast<cudaStream_t>(stream), bk, l->d_claim);
  if (e != cudaSuccess) return cuda_err(e, "tf_pack_buckets launch");
  l->seq = bk.seq;
  e = note_table_use(l, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_err(e, "cudaEventRecord(bucket table use)");
  return FG_OK;
}
}  // namespace

fg_status tf_pack_buckets(tf_layout* l, float scale, void* buf, void* stream) {
  return pack_buckets(l, scale, buf, stream, nullptr, 0, 0);
}

fg_status tf_pack_buckets_observed(tf_layout* l, float scale, void* buf, uint64_t* times, uint32_t seq_offset,
                                   int64_t wait_limit_ns, void* stream) {
  if (!times) return err(FG_EINVAL, "null argument");
  if (reinterpret_cast<uintptr_t>(times) % 8) return err(FG_EINVAL, "times must be 8-byte aligned");
  if (wait_limit_ns <= 0) return err(FG_EINVAL, "wait_limit_ns must be positive");
  if (l && l->nb) {
    // the packing CTAs' finishing time is a maximum: it starts from zero
    cudaError_t e = cudaMemsetAsync(times + l->nb, 0, sizeof(uint64_t), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_err(e, "cudaMemsetAsync(observed times)");
  }
  return pack_buckets(l, scale, buf, stream, times, seq_offset, wait_limit_ns);
}

fg_status tf_bucket_wait(tf_layout* l, int32_t b, void* stream) {
  if (!l) return err(FG_EINVAL, "null argument");
  if (!l->nb || !l->seq) return err(FG_EINVAL, "no bucketed pack has been enqueued");
  if (b < 0 || b >= l->nb) return err(FG_EINVAL, "bucket out of range");
  WaitValueFn fn = wait_value_fn();
  if (!fn) return err(FG_EUNSUPPORTED, "cuStreamWaitValue32 is not available");
  // the count reaches this pack's total (a cyclic comparison, as the count
  // wraps modulo 2^32)
  const int32_t* count = l->d_bucket + l->nchunks + l->nb + b;
  const uint32_t target = l->seq * l->bucket_chunks[b];
  CUresult r = fn(static_cast<CUstream>(stream), reinterpret_cast<CUdeviceptr>(count), target, CU_STREAM_WAIT_VALUE_GEQ);
  if (r != CUDA_SUCCESS) return err(FG_ECUDA, "cuStreamWaitValue32 failed (" + std::to_string((int)r) + ")");
  const cudaError_t e = note_table_use(l, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_err(e, "cudaEventRecord(bucket table use)");
  return FG_OK;
}

fg_status tf_bucket_ready(const tf_layout* l, int32_t b, int32_t* ready) {
  if (!l || !ready) return err(FG_EINVAL, "null argument");
  if (!l->nb || !l->seq) return err(FG_EINVAL, "no bucketed pack has been enqueued");
  if (b < 0 || b >= l->nb) return err(FG_EINVAL, "bucket out of range");
  uint32_t v = 0;
  cudaError_t e = cudaMemcpy(&v, l->d_bucket + l->nchunks + l->nb + b, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_err(e, "reading a bucket's count");
  *ready = (int32_t)(v - l->seq * l->bucket_chunks[b]) >= 0 ? 1 : 0;
  return FG_OK;
}

fg_status tf_unpack(const tf_layout* l, float uscale, const void* buf, void* stream) {
  if (!l) return err(FG_EINVAL, "null argument");
  return tf_unpack_range(l, 0, l->n, uscale, buf, stream);
}

// Threshold fusion in production order: a tensor joins the open bucket while
// the bucket's padded bytes stay within the threshold, otherwise it opens
// the next one (a tensor above the threshold sits alone).
fg_status tf_plan_threshold(int32_t n, const int64_t* numel, fg_dtype buf_dtype, int64_t align,
                            int64_t threshold, int32_t* bounds, int32_t* n_buckets) {
  if (n < 0 || (n > 0 && !numel) || !bounds || !n_buckets) return err(FG_EINVAL, "null argument");
  if (buf_dtype != FG_BF16 && buf_dtype != FG_F32) return err(FG_EINVAL, "unknown buffer dtype");
  if (align < 16 || (align & (align - 1))) return err(FG_EINVAL, "align_bytes must be a power of two >= 16");
  if (threshold < 0) return err(FG_EINVAL, "negative threshold");
  const int64_t eb = buf_dtype == FG_BF16 ? 2 : 4;
  int32_t nb = 0;
  bounds[0] = 0;
  int64_t cur = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (numel[i] < 0) return err(FG_ESHAPE, "negative element count");
    const int64_t sz = round_up(numel[i] * eb, align);
    if (i > bounds[nb] && cur + sz > threshold) {
      bounds[++nb] = i;
      cur = 0;
    }
    cur += sz;
  }
  if (n > 0) bounds[++nb] = n;
  *n_buckets = nb;
  return FG_OK;
}

fg_status tf_buckets_merge(int32_t* bounds, int32_t* n_buckets, int32_t j) {
  if (!bounds || !n_buckets) return err(FG_EINVAL, "null argument");
  if (j < 0 || j + 1 >= *n_buckets) return err(FG_EINVAL, "bucket has no successor");
  for (int32_t k = j + 1; k < *n_buckets; ++k) bounds[k] = bounds[k + 1];
  --*n_buckets;
  return FG_OK;
}

fg_status tf_sync_status(tf_layout* l, void* stream) {
  if (!l) return err(FG_EINVAL, "null layout");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize");
  int32_t flag = 0;
  e = cudaMemcpy(&flag, l->d_err, sizeof(flag), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_err(e, "reading the device error flag");
  if (flag == 0) return FG_OK;
  cudaMemset(l->d_err, 0, sizeof(int32_t));
  if (flag == DEVERR_TIMEOUT) return err(FG_ETIMEOUT, "a device-side wait expired (a chunk load or a watched bucket)");
  return err(FG_EDEVICE, "device error flag " + std::to_string(flag));
}

void tf_layout_destroy(tf_layout* l) {
  if (!l) return;
  if (l->d_bucket) l->retired.push_back(tf_layout::Retired{l->d_bucket, std::move(l->users)});
  free_retired(l, true);
  if (l->d_chunks) cudaFree(l->d_chunks);
  delete l;
}

}  // extern "C"
