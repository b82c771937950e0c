// Group compilation: one operator program per group, evaluated in the frame
// of the group's output (TVM "Operator Fusion", FuseTIR: the operators of a
// group merge into one function whose intermediates never reach global
// memory).  Every operator is evaluated at the frame point; injective
// operators turn into index maps on the leaves they read (a transpose or
// reshape moves no data inside a group), broadcasts read their vector at the
// mapped row or column.
#include <algorithm>
#include <map>
#include <tuple>

#include "host.h"

namespace fg {

bool Map::operator==(const Map& o) const {
  if (n != o.n || shift != o.shift) return false;
  for (int k = 0; k < n; ++k)
    if (d[k] != o.d[k] || m[k] != o.m[k] || s[k] != o.s[k]) return false;
  return true;
}

namespace {

[[noreturn]] void fail(fg_status st, const std::string& msg) { throw CompileError{st, msg}; }

struct Term { int64_t d, m, s; };

Map make_map(std::vector<Term> t) {
  // drop unit digits, order by place value, merge digits that continue
  // each other both in the frame index and in the value index
  t.erase(std::remove_if(t.begin(), t.end(), [](const Term& x) { return x.m == 1; }), t.end());
  std::sort(t.begin(), t.end(), [](const Term& a, const Term& b) { return a.s < b.s; });
  std::vector<Term> out;
  for (const Term& x : t) {
    if (!out.empty() && out.back().s * out.back().m == x.s && out.back().d * out.back().m == x.d) {
      out.back().m *= x.m;
    } else {
      out.push_back(x);
    }
  }
  if ((int)out.size() > kMaxTerms) fail(FG_EUNSUPPORTED, "index map needs more than 4 digits");
  Map mp;
  mp.n = (int)out.size();
  for (int k = 0; k < mp.n; ++k) {
    mp.d[k] = out[k].d;
    mp.m[k] = out[k].m;
    mp.s[k] = out[k].s;
  }
  return mp;
}

std::vector<Term> terms(const Map& mp) {
  std::vector<Term> t;
  for (int k = 0; k < mp.n; ++k) t.push_back({mp.d[k], mp.m[k], mp.s[k]});
  return t;
}

Map ident(int64_t rows, int64_t cols) { return make_map({{1, rows * cols, 1}}); }

// f % Q and f / Q as maps; Q must fall on a digit boundary (a digit may be
// split when its radix divides accordingly).
void split(const Map& mp, int64_t Q, Map& lo, Map& hi) {
  std::vector<Term> L, H;
  for (Term t : terms(mp)) {
    if (t.s * t.m <= Q) {
      L.push_back(t);
    } else if (t.s >= Q) {
      if (t.s % Q) fail(FG_EUNSUPPORTED, "index map does not split at the row boundary");
      H.push_back({t.d, t.m, t.s / Q});
    } else {
      int64_t q = Q / t.s;
      if (Q % t.s || t.m % q) fail(FG_EUNSUPPORTED, "index map does not split at the row boundary");
      L.push_back({t.d, q, t.s});
      H.push_back({t.d * q, t.m / q, 1});
    }
  }
  int64_t prod = 1;
  for (const Term& t : L) prod *= t.m;
  if (!H.empty() && prod != Q) fail(FG_EUNSUPPORTED, "index map does not split at the row boundary");
  lo = make_map(L);
  hi = make_map(H);
  lo.shift = hi.shift = mp.shift;
}

// The map of x = y^T's index, given y's map; x is [A, B], y is [B, A]:
// f_x = (f_y % A) * B + f_y / A.
Map transpose_map(const Map& fy, int64_t A, int64_t B) {
  Map lo, hi;
  split(fy, A, lo, hi);
  std::vector<Term> t;
  for (Term x : terms(lo)) t.push_back({x.d, x.m, x.s * B});
  for (Term x : terms(hi)) t.push_back(x);
  Map r = make_map(t);
  r.shift = fy.shift;
  return r;
}

// The class of a map's digits (its shift aside).
int classify(const Map& shifted, int64_t FR, int64_t FC) {
  Map mp = shifted;
  mp.shift = 0;
  if (mp == ident(FR, FC)) return LEAF_IDENT;
  if (mp == make_map({{FC, FR, 1}, {1, FC, FR}})) return LEAF_TRANS;
  if (mp == make_map({{1, FC, 1}})) return LEAF_COL;
  if (mp == make_map({{FC, FR, 1}})) return LEAF_ROW;
  return LEAF_GATHER;
}

// ---- expression DAG --------------------------------------------------------

enum ExprKind { E_LEAF, E_ACC, E_UN, E_BIN, E_SEL };

struct Expr {
  ExprKind kind;
  int vm;                // VmOp for E_UN / E_BIN
  float imm = 0.f;
  int a = -1, b = -1;    // children
  int leaf = -1;         // index into leaves (E_LEAF)
  int uses = 0;
  int need = 1;          // registers to evaluate (Sethi-Ullman, no caching)
};

struct Builder {
  const Graph& g;
  std::vector<char> in_group;     // per node
  int anchor = -1;                // node read as the accumulator (matmul / reduce)
  Map anchor_map;
  int64_t FR, FC;
  std::vector<Expr> ex;
  std::vector<LeafUse> leaves;
  std::map<std::tuple<int, int, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t,
                      int64_t, int64_t, int64_t, int64_t, int64_t, int64_t>, int> memo;
  bool tuples_ok = true;          // the epilogue of a reduce or matmul group has no tuples

  Builder(const Graph& gg, const std::vector<int32_t>& nodes, int64_t fr, int64_t fc)
      : g(gg), in_group(gg.nodes.size(), 0), FR(fr), FC(fc) {
    for (int x : nodes) in_group[x] = 1;
  }

  int mk(Expr e) {
    ex.push_back(e);
    return (int)ex.size() - 1;
  }

  int leaf(int value, const Map& mp) {
    for (size_t i = 0; i < leaves.size(); ++i)
      if (leaves[i].value == value && leaves[i].map == mp) return (int)i;
    leaves.push_back({value, mp, classify(mp, FR, FC), g.values[value].numel()});
    return (int)leaves.size() - 1;
  }

  int build(int value, const Map& mp) {
    auto key = std::make_tuple(value, mp.n, mp.d[0], mp.m[0], mp.s[0], mp.d[1], mp.m[1], mp.s[1],
                               mp.d[2], mp.m[2], mp.s[2], mp.d[3], mp.m[3], mp.s[3], mp.shift);
    auto it = memo.find(key);
    if (it != memo.end()) {
      ex[it->second].uses++;
      return it->second;
    }
    int id = build_new(value, mp);
    ex[id].uses++;
    memo[key] = id;
    built.push_back({value, mp, id});
    return id;
  }

  struct Built {
    int value;
    Map map;
    int expr;
  };
  std::vector<Built> built;   // every (value, map) evaluated, in build order

  // Expressions for the group's extra outputs, appended to the DAG: each at a
  // map the main program already evaluates it at when that map covers all its
  // elements, else at the frame's flat index (any one-to-one map will do for
  // a value nothing else in the group reads).
  void add_xouts(CompiledGroup& cg) {
    for (int32_t v : cg.xout_values) {
      const Value& xv = g.values[v];
      if (xv.numel() != FR * FC) fail(FG_EUNSUPPORTED, "an extra output must have as many elements as the frame");
      int expr = -1;
      Map mp;
      for (const Built& b : built)
        if (b.value == v) {
          expr = b.expr;
          mp = b.map;
          break;
        }
      if (expr < 0) {
        mp = ident(FR, FC);
        expr = build(v, mp);
      }
      int cls = classify(mp, FR, FC);
      if (cls != LEAF_IDENT && cls != LEAF_TRANS) {
        cls = LEAF_GATHER;
        if (FR * FC >= (int64_t)1 << 31) fail(FG_EUNSUPPORTED, "a permuted extra output of a frame of 2^31 or more elements");
      }
      cg.xout_maps.push_back(mp);
      cg.xout_cls.push_back(cls);
      cg.xout_expr.push_back(expr);
    }
  }

  int build_new(int value, const Map& mp) {
    const Value& v = g.values[value];
    int nd = v.node;
    if (nd < 0 || !in_group[nd]) {
      Expr e{E_LEAF, 0};
      e.leaf = leaf(value, mp);
      return mk(e);
    }
    if (nd == anchor) {
      if (!(mp == anchor_map)) fail(FG_EUNSUPPORTED, "accumulator read at a moved index");
      return mk(Expr{E_ACC, VM_PUSH_ACC});
    }
    const Node& n = g.nodes[nd];
    auto un = [&](int vm, int a, float imm) {
      Expr e{E_UN, vm};
      e.a = a;
      e.imm = imm;
      return mk(e);
    };
    auto bin = [&](int vm, int a, int b) {
      Expr e{E_BIN, vm};
      e.a = a;
      e.b = b;
      return mk(e);
    };
    auto arg = [&](int i) { return n.args[i]; };
    const Value& x0 = g.values[arg(0)];
    switch (n.op) {
      case FG_OP_CONCAT:
        return build_alias(arg(0), mp);   // a tuple's value is already its fields stacked
      case FG_OP_TUPLE: {
        // the tuple's row for the frame point: the frame row when the tuple
        // is in the frame's layout, the frame column when it is transposed
        if (!tuples_ok) fail(FG_EUNSUPPORTED, "a tuple in a reduce or matmul epilogue");
        if (mp.shift) fail(FG_EUNSUPPORTED, "a tuple read through another tuple's field");
        const Value& tv = g.values[n.value];
        const int cls = classify(mp, FR, FC);
        int axis;
        if (cls == LEAF_IDENT && tv.cols == FC) axis = 0;
        else if (cls == LEAF_TRANS && tv.cols == FR) axis = 1;
        else fail(FG_EUNSUPPORTED, "a tuple read through a map other than the frame's layout or its transpose");
        std::vector<int> fields;
        std::vector<int64_t> bounds;
        int64_t off = 0;
        for (int32_t f : n.args) {
          Map fm = mp;
          fm.shift = axis == 0 ? off * tv.cols : off;   // the field's rows start `off` rows down
          fields.push_back(build(f, fm));
          off += g.values[f].rows;
          bounds.push_back(off);
        }
        if (off >= (int64_t)1 << 31) fail(FG_EUNSUPPORTED, "tuple too tall");
        int acc = fields.back();
        for (int k = (int)fields.size() - 2; k >= 0; --k) {
          Expr e{E_SEL, axis};
          e.a = fields[k];
          e.b = acc;
          e.leaf = (int)bounds[k];
          acc = mk(e);
        }
        return acc;
      }
      case FG_OP_TRANSPOSE:
        return build_alias(arg(0), transpose_map(mp, x0.rows, x0.cols));
      case FG_OP_RESHAPE:
      case FG_OP_OPAQUE_COPY:
        return build_alias(arg(0), mp);
      case FG_OP_ADD: {
        int acc = bin(VM_ADD, build(arg(0), mp), build(arg(1), mp));
        for (size_t i = 2; i < n.args.size(); ++i) {
          ex[acc].uses++;
          acc = bin(VM_ADD, acc, build(arg((int)i), mp));
        }
        return acc;
      }
      case FG_OP_SUB: return bin(VM_SUB, build(arg(0), mp), build(arg(1), mp));
      case FG_OP_MUL: return bin(VM_MUL, build(arg(0), mp), build(arg(1), mp));
      case FG_OP_DIV: return bin(VM_DIV, build(arg(0), mp), build(arg(1), mp));
      case FG_OP_SCALE: return un(VM_SCALE, build(arg(0), mp), n.attrs[0]);
      case FG_OP_ADDC: return un(VM_ADDC, build(arg(0), mp), n.attrs[0]);
      case FG_OP_RELU: return un(VM_RELU, build(arg(0), mp), 0.f);
      case FG_OP_EXP: return un(VM_EXP, build(arg(0), mp), 0.f);
      case FG_OP_SIGMOID: return un(VM_SIGMOID, build(arg(0), mp), 0.f);
      case FG_OP_TANH: return un(VM_TANH, build(arg(0), mp), 0.f);
      case FG_OP_NEG: return un(VM_NEG, build(arg(0), mp), 0.f);
      case FG_OP_BADD_COL:
      case FG_OP_BMUL_COL:
      case FG_OP_BADD_ROW:
      case FG_OP_BMUL_ROW: {
        bool col = n.op == FG_OP_BADD_COL || n.op == FG_OP_BMUL_COL;
        Map lo, hi;
        split(mp, x0.cols, lo, hi);
        int xa = build(arg(0), mp);
        int va = build(arg(1), col ? lo : hi);
        bool add = n.op == FG_OP_BADD_COL || n.op == FG_OP_BADD_ROW;
        return bin(add ? VM_ADD : VM_MUL, xa, va);
      }
      default:
        fail(FG_EUNSUPPORTED, "operator cannot sit inside a group program");
    }
  }

  // Injective operators add no instruction: the operand's expression is the
  // result.  Its use count is bumped by the caller's `build`.
  int build_alias(int value, const Map& mp) {
    int id = build(value, mp);
    ex[id].uses--;
    return id;
  }
};

// ---- postfix emission --------------------------------------------------------

struct Emitter {
  std::vector<Expr>& ex;
  std::vector<VmInstr> code;
  int depth = 0, max_depth = 0, max_slot = 0;
  std::vector<int> slot_of;     // expr -> slot or -1
  std::vector<int> remaining;   // references still to emit
  std::vector<char> slot_busy;

  explicit Emitter(std::vector<Expr>& e)
      : ex(e), slot_of(e.size(), -1), remaining(e.size(), 0), slot_busy(kMaxSlots, 0) {
    for (size_t i = 0; i < e.size(); ++i) remaining[i] = e[i].uses;
    for (size_t i = 0; i < e.size(); ++i) need(i);
  }

  int need(size_t i) {
    Expr& e = ex[i];
    if (e.kind == E_UN) e.need = ex[e.a].need;
    if (e.kind == E_BIN) {
      int la = ex[e.a].need, lb = ex[e.b].need;
      e.need = la == lb ? la + 1 : std::max(la, lb);
    }
    return e.need;
  }

  void put(int op, int slot = 0, int arg = 0, float imm = 0.f) {
    if ((int)code.size() >= kMaxProg) fail(FG_EUNSUPPORTED, "group program too long");
    code.push_back(VmInstr{(uint16_t)vm_case(op, depth, slot), (uint16_t)arg, imm});
  }
  void push_depth() {
    ++depth;
    if (depth > kMaxDepth) fail(FG_EUNSUPPORTED, "group program needs more than 8 stack registers");
    max_depth = std::max(max_depth, depth);
  }
  int alloc_slot() {
    for (int s = 0; s < kMaxSlots; ++s)
      if (!slot_busy[s]) {
        slot_busy[s] = 1;
        max_slot = std::max(max_slot, s + 1);
        return s;
      }
    return -1;
  }
  // a value that can be the right operand of a binary op without a push
  bool direct(int i) const { return ex[i].kind == E_LEAF || slot_of[i] >= 0; }
  void use_slot(int i) {
    if (--remaining[i] == 0) slot_busy[slot_of[i]] = 0;
  }

  // Emit code that leaves expr i on top of the stack.
  void emit(int i) {
    Expr& e = ex[i];
    if (slot_of[i] >= 0) {
      put(VM_PUSH_SLOT, slot_of[i]);
      push_depth();
      use_slot(i);
      return;
    }
    switch (e.kind) {
      case E_LEAF:
        put(VM_PUSH_LEAF, 0, e.leaf);
        push_depth();
        return;   // leaves are re-read from shared memory, never kept in slots
      case E_ACC:
        put(VM_PUSH_ACC);
        push_depth();
        break;
      case E_UN:
        emit(e.a);
        put(e.vm, 0, 0, e.imm);
        break;
      case E_BIN: {
        int a = e.a, b = e.b;
        const bool comm = e.vm == VM_ADD || e.vm == VM_MUL;
        if (comm && (direct(a) && !direct(b))) std::swap(a, b);
        else if (comm && !direct(b) && ex[b].need > ex[a].need) std::swap(a, b);
        const int off = e.vm - VM_ADD;
        if (direct(b)) {
          emit(a);
          if (ex[b].kind == E_LEAF) {
            put(VM_ADD_L + off, 0, ex[b].leaf);
          } else {
            put(VM_ADD_S + off, slot_of[b]);
            use_slot(b);
          }
          break;
        }
        // evaluate a deep right operand into a slot first if the stack
        // would overflow otherwise
        if (depth + std::max(ex[a].need, ex[b].need + 1) > kMaxDepth) {
          int spill = alloc_slot();
          if (spill >= 0) {
            emit(b);
            put(VM_STORE, spill);
            --depth;
            emit(a);
            put(VM_ADD_S + off, spill);
            slot_busy[spill] = 0;
            break;
          }
        }
        emit(a);
        emit(b);
        put(e.vm);
        --depth;
        break;
      }
    }
    // a value needed again later is kept in a save slot until its last use
    if (--remaining[i] > 0) {
      int s = alloc_slot();
      if (s < 0) fail(FG_EUNSUPPORTED, "group program keeps more than 8 values live");
      slot_of[i] = s;
      put(VM_TEE, s);
    }
  }
};

struct Program {
  std::vector<VmInstr> code;
  std::vector<LeafUse> leaves;
  int depth = 0, slots = 0;
  std::vector<JExpr> dag;
  int root = -1;
  bool needs_jit = false;
};

Program emit_program(Builder& b, int root) {
  Program p;
  for (const Expr& e : b.ex) p.dag.push_back(JExpr{(int)e.kind, e.vm, e.imm, e.a, e.b, e.leaf});
  p.root = root;
  p.leaves = b.leaves;
  for (const Expr& e : b.ex)
    if (e.kind == E_SEL) {
      // selects run in compiled programs only: no interpreter program
      p.needs_jit = true;
      if ((int)p.leaves.size() > kMaxLeaves) fail(FG_EUNSUPPORTED, "group reads more than 24 leaf views");
      return p;
    }
  p.root = root;
  Emitter em(b.ex);
  em.emit(root);
  if (em.depth != 1) fail(FG_EUNSUPPORTED, "internal: unbalanced program");
  p.code = em.code;
  p.leaves = b.leaves;
  p.depth = em.max_depth;
  p.slots = em.max_slot;
  if ((int)p.leaves.size() > kMaxLeaves) fail(FG_EUNSUPPORTED, "group reads more than 24 leaf views");
  return p;
}

}  // namespace

CompiledGroup compile_group(const Graph& g, const std::vector<int32_t>& nodes_in) {
  CompiledGroup cg;
  cg.nodes = nodes_in;
  std::sort(cg.nodes.begin(), cg.nodes.end());
  // the sink: the last member whose value no other member reads (for
  // FuseOps groups, the last member; a copied operator made by duplicate
  // fusion sits after its reader and is never the sink)
  {
    std::vector<char> read_in(g.values.size(), 0);
    for (int x : cg.nodes)
      for (int32_t a : g.nodes[x].args) read_in[a] = 1;
    cg.sink = -1;
    for (int x : cg.nodes)
      if (!read_in[g.nodes[x].value]) cg.sink = x;
    if (cg.sink < 0) fail(FG_EUNSUPPORTED, "internal: group without a sink");
  }
  cg.out_value = g.nodes[cg.sink].value;
  int mm = -1, red = -1;
  for (int x : cg.nodes) {
    int op = g.nodes[x].op;
    if (op == FG_OP_MATMUL_BF16) {
      if (mm >= 0) fail(FG_EUNSUPPORTED, "two matmuls in one group");
      mm = x;
    }
    if (op == FG_OP_ROWSUM || op == FG_OP_ROWMAX) {
      if (red >= 0) fail(FG_EUNSUPPORTED, "two reductions in one group");
      red = x;
    }
  }
  if (mm >= 0 && red >= 0) fail(FG_EUNSUPPORTED, "matmul and reduction in one group");

  // distinct outside values, first-use order
  std::vector<char> in(g.nodes.size(), 0);
  for (int x : cg.nodes) in[x] = 1;
  // values of the group read outside it (non-duplicate fusion of an operator
  // whose output other operators still need) or marked as graph outputs
  {
    std::vector<char> read_out(g.values.size(), 0);
    for (size_t x = 0; x < g.nodes.size(); ++x)
      if (!in[x])
        for (int32_t a : g.nodes[x].args) read_out[a] = 1;
    std::vector<char> read_in(g.values.size(), 0);
    for (int x : cg.nodes)
      for (int32_t a : g.nodes[x].args) read_in[a] = 1;
    for (int x : cg.nodes) {
      const int32_t v = g.nodes[x].value;
      if (v != cg.out_value && (read_out[v] || g.is_output[v] || !read_in[v])) cg.xout_values.push_back(v);
    }
    if ((int)cg.xout_values.size() > kMaxXOut) fail(FG_EUNSUPPORTED, "more than 4 extra outputs in one group");
    if (!cg.xout_values.empty() && mm >= 0) fail(FG_EUNSUPPORTED, "extra outputs of a matmul group");
    if (!cg.xout_values.empty() && red >= 0) {
      // only values of the prologue (frame-shaped, before the reduction)
      std::vector<char> after(g.nodes.size(), 0);
      after[red] = 1;
      for (int x : cg.nodes)
        for (int32_t a : g.nodes[x].args) {
          const int prod = g.values[a].node;
          if (prod >= 0 && in[prod] && after[prod]) after[x] = 1;
        }
      for (int32_t v : cg.xout_values)
        if (after[g.values[v].node]) fail(FG_EUNSUPPORTED, "an extra output after the reduction");
    }
  }
  for (int x : cg.nodes)
    for (int32_t a : g.nodes[x].args) {
      int prod = g.values[a].node;
      if (prod >= 0 && in[prod]) continue;
      if (std::find(cg.leaf_values.begin(), cg.leaf_values.end(), a) == cg.leaf_values.end())
        cg.leaf_values.push_back(a);
    }
  for (int32_t a : cg.leaf_values) {
    if (g.values[a].dtype != FG_F32 && !(mm >= 0 && (a == g.nodes[mm].args[0] || a == g.nodes[mm].args[1])))
      fail(FG_EUNSUPPORTED, "bf16 value read outside a matmul operand");
    cg.alg_bytes += g.values[a].bytes();
  }
  const Value& out = g.values[cg.out_value];
  cg.alg_bytes += out.bytes();
  for (int32_t v : cg.xout_values) cg.alg_bytes += g.values[v].bytes();

  if (mm >= 0) {
    const Node& n = g.nodes[mm];
    cg.exec = FG_EXEC_GEMM;
    cg.mm_a = n.args[0];
    cg.mm_b = n.args[1];
    cg.mm_ta = n.attrs.size() > 0 ? (int)n.attrs[0] : 0;
    cg.mm_tb = n.attrs.size() > 1 ? (int)n.attrs[1] : 0;
    const Value& mv = g.values[n.value];
    cg.M = mv.rows;
    cg.N = mv.cols;
    const Value& A = g.values[cg.mm_a];
    cg.K = cg.mm_ta ? A.rows : A.cols;
    cg.alg_flops = 2 * cg.M * cg.N * cg.K;
    cg.FR = cg.M;
    cg.FC = cg.N;
    // the epilogue runs on the accumulator tile; operands are not leaves of it
    Builder b(g, cg.nodes, cg.FR, cg.FC);
    b.anchor = mm;
    b.anchor_map = ident(cg.FR, cg.FC);
    b.tuples_ok = false;
    Program p = emit_program(b, b.build(cg.out_value, ident(cg.FR, cg.FC)));
    cg.prog = p.code;
    cg.leaves = p.leaves;
    cg.depth = p.depth;
    cg.slots = p.slots;
    cg.dag = p.dag;
    cg.dag_root = p.root;
    for (auto& l : cg.leaves)
      if (l.value == cg.mm_a || l.value == cg.mm_b) fail(FG_EUNSUPPORTED, "matmul operand read by the epilogue");
    return cg;
  }
  if (red >= 0) {
    const Node& n = g.nodes[red];
    cg.exec = FG_EXEC_REDUCE;
    cg.red_op = n.op == FG_OP_ROWSUM ? RED_SUM : RED_MAX;
    const Value& x = g.values[n.args[0]];
    if (x.ndim != 2) fail(FG_ESHAPE, "row reduction of a rank-1 value");
    cg.FR = x.rows;
    cg.FC = x.cols;
    Builder b(g, cg.nodes, cg.FR, cg.FC);
    b.anchor = red;   // never reached from the prologue root
    b.anchor_map = ident(1, cg.FR);
    const int root = b.build(n.args[0], ident(cg.FR, cg.FC));
    b.add_xouts(cg);
    Program p = emit_program(b, root);
    cg.prog = p.code;
    cg.leaves = p.leaves;
    cg.depth = p.depth;
    cg.slots = p.slots;
    cg.dag = p.dag;
    cg.dag_root = p.root;
    cg.needs_jit = p.needs_jit;
    if (cg.sink != red) {
      // epilogue on the reduced vector (allow_reduce_epilogue)
      Builder be(g, cg.nodes, 1, cg.FR);
      be.anchor = red;
      be.anchor_map = ident(1, cg.FR);
      be.tuples_ok = false;
      Program pe = emit_program(be, be.build(cg.out_value, ident(1, cg.FR)));
      if ((int)pe.code.size() > kMaxEpi) fail(FG_EUNSUPPORTED, "reduce epilogue too long");
      if ((int)pe.leaves.size() > kMaxEpiLeaves) fail(FG_EUNSUPPORTED, "reduce epilogue reads too many values");
      for (auto& l : pe.leaves)
        if (l.cls != LEAF_IDENT) fail(FG_EUNSUPPORTED, "reduce epilogue reads a moved vector");
      cg.epi = pe.code;
      cg.epi_dag = pe.dag;
      cg.epi_root = pe.root;
      for (auto& l : pe.leaves) cg.epi_leaf_values.push_back(l.value);
      cg.epi_depth = pe.depth;
      cg.epi_slots = pe.slots;
    }
    return cg;
  }
  cg.exec = FG_EXEC_ELEMWISE;
  cg.FR = out.rows;
  cg.FC = out.cols;
  Builder b(g, cg.nodes, cg.FR, cg.FC);
  const int root = b.build(cg.out_value, ident(cg.FR, cg.FC));
  b.add_xouts(cg);
  Program p = emit_program(b, root);
  cg.prog = p.code;
  cg.leaves = p.leaves;
  cg.depth = p.depth;
  cg.slots = p.slots;
  cg.dag = p.dag;
  cg.dag_root = p.root;
  cg.needs_jit = p.needs_jit;
  return cg;
}

// Which leaves are staged through shared memory by TMA, and the pipeline
// depth.  A TMA tensor needs 16-byte row strides, so IDENT leaves need a
// frame width that is a multiple of 4 floats and TRANS leaves a frame height
// that is.  Everything else is gathered from global memory.
void plan_staging(const Graph& g, CompiledGroup& cg, const BuildOpts& o) {
  (void)g;
  const bool gemm = cg.exec == FG_EXEC_GEMM;
  const int TR = gemm ? 128 : kTileR, TC = gemm ? 32 : kTileC;
  auto box_bytes = [&](int cls) -> int {
    switch (cls) {
      case LEAF_IDENT: case LEAF_TRANS: return TR * TC * 4;
      case LEAF_COL: return TC * 4;
      case LEAF_ROW: return TR * 4;
      default: return 0;
    }
  };
  const bool rows_ok = cg.FC % 4 == 0 || cg.FR == 1;
  const bool cols_ok = cg.FR % 4 == 0 || cg.FC == 1;
  // output: 1 = CTA tile staged in smem + TMA store, 2 = per-warp slices
  // stored by TMA, 0 = direct stores
  const int omode = (o.flags >> 24) & 3;
  cg.out_tma = (rows_ok && cg.exec == FG_EXEC_ELEMWISE) ? (omode == 0 ? 2 : omode == 3 ? 0 : omode) : 0;
  std::vector<char> stage(cg.leaves.size(), 0);
  int want = 0;
  for (size_t i = 0; i < cg.leaves.size(); ++i) {
    int c = cg.leaves[i].cls;
    bool ok = (c == LEAF_IDENT && rows_ok) || (c == LEAF_TRANS && cols_ok) || c == LEAF_COL || c == LEAF_ROW;
    // a shifted leaf (a tuple's field) moves its boxes by whole rows and
    // columns; a copy's innermost coordinate must stay 16-byte aligned
    const int64_t sh = cg.leaves[i].map.shift;
    if (sh) {
      const int64_t sr = sh / cg.FC, sc = sh % cg.FC;
      const int64_t inner = (c == LEAF_IDENT || c == LEAF_COL) ? sc : sr;
      if (gemm || inner % 4) ok = false;
    }
    if (ok && want < kMaxStaged) {
      stage[i] = 1;
      ++want;
    }
  }
  // big boxes first (1024-byte aligned for the 128-byte swizzle), then vectors
  auto layout = [&](std::vector<int>* offs) {
    int off = 0;
    for (size_t i = 0; i < cg.leaves.size(); ++i)
      if (stage[i] && box_bytes(cg.leaves[i].cls) >= 1024) {
        if (offs) (*offs)[i] = off;
        off += box_bytes(cg.leaves[i].cls);
      }
    for (size_t i = 0; i < cg.leaves.size(); ++i)
      if (stage[i] && box_bytes(cg.leaves[i].cls) < 1024) {
        if (offs) (*offs)[i] = off;
        off += (box_bytes(cg.leaves[i].cls) + 127) / 128 * 128;
      }
    return (off + 1023) / 1024 * 1024;
  };
  int fixed = 2048;   // barriers + alignment slack
  // extra outputs with identity or transposed maps go out like the sink
  // output: per-warp slices in shared memory, one TMA store each
  cg.xout_tma = 0;
  if (cg.exec == FG_EXEC_ELEMWISE && cg.out_tma == 2 && !cg.xout_values.empty()) {
    cg.xout_tma = 1;
    for (int c : cg.xout_cls)
      if (!((c == LEAF_IDENT && rows_ok) || (c == LEAF_TRANS && cols_ok && cg.FR % 4 == 0))) cg.xout_tma = 0;
  }
  if (!gemm) {
    if (cg.out_tma) fixed += 3 * TR * TC * 4;               // three output buffers (per CTA or per warp)
    if (cg.xout_tma) fixed += 3 * (int)cg.xout_values.size() * TR * TC * 4;   // and per extra output
    if (cg.exec == FG_EXEC_REDUCE) fixed += 2 * kConsumerWarps * 32 * 4;   // double-buffered row partials
  }
  // dynamic shared memory per CTA; about 5 KB of static tables come on top
  const int budget_two = 106 * 1024, budget_one = 218 * 1024;
  int sb = layout(nullptr);
  int budget = budget_two;
  if (!gemm) {
    while (true) {
      if (sb == 0 || (budget_two - fixed) / sb >= 3) { budget = budget_two; break; }
      if ((budget_one - fixed) / sb >= 2) { budget = budget_one; break; }
      int last = -1;   // demote the last staged leaf to a gather
      for (size_t i = 0; i < cg.leaves.size(); ++i) if (stage[i]) last = (int)i;
      stage[last] = 0;
      sb = layout(nullptr);
    }
  } else {
    // GEMM epilogue: several buffers of staged leaves must fit beside the
    // operand pipeline; demote leaves beyond 40 KB per chunk
    while (sb > 40 * 1024) {
      int last = -1;
      for (size_t i = 0; i < cg.leaves.size(); ++i) if (stage[i]) last = (int)i;
      stage[last] = 0;
      sb = layout(nullptr);
    }
  }
  if (cg.FR * cg.FC >= (int64_t(1) << 31))
    for (size_t i = 0; i < cg.leaves.size(); ++i)
      if (!stage[i]) throw CompileError{FG_EUNSUPPORTED, "gathered leaf in a frame of 2^31 or more elements"};
  cg.leaf_stage_off.assign(cg.leaves.size(), -1);
  cg.stage_bytes = layout(&cg.leaf_stage_off);
  cg.nstaged = cg.ngathered = 0;
  for (size_t i = 0; i < cg.leaves.size(); ++i) {
    if (stage[i]) {
      cg.nstaged++;
    } else {
      cg.leaves[i].cls = LEAF_GATHER;
      cg.ngathered++;
    }
  }
  if (!gemm) {
    int ns = cg.stage_bytes ? (budget - fixed) / cg.stage_bytes : 4;
    // an even depth: each of the two producers owns every other ring slot
    cg.nstages = std::max(2, std::min(ns, kMaxStages)) & ~1;
    cg.smem_bytes = fixed + cg.nstages * cg.stage_bytes;
    cg.ctas_per_sm = budget == budget_two ? 2 : 1;
  }
}

}  // namespace fg
