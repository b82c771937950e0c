// Pattern annotation, post-dominator tree and FuseOps-style grouping.
//
// TVM "Operator Fusion": Operator Pattern Classification (kinds and their
// order, CombinePattern = max); FuseOps > Algorithm steps 1-3 (forward graph,
// post-dominator tree by LCA on the DAG, CheckPath + CommitFuse with
// union-find); Fusion rules (phases 0, 1 and 2, reduce only as a sink,
// opaque barrier, kMaxFusedOps and the argument limit).  A tuple fuses like an
// injective operator in phase 1 and, once merged with other operators, counts
// as injective in its group's pattern; phase 2 fuses injective-or-simpler
// producers into a tuple that a later group has absorbed.
#include <algorithm>

#include "host.h"

namespace fg {

Kind op_kind(int op) {
  switch (op) {
    case FG_OP_ADD: case FG_OP_SUB: case FG_OP_MUL: case FG_OP_DIV:
    case FG_OP_SCALE: case FG_OP_ADDC: case FG_OP_RELU: case FG_OP_EXP:
    case FG_OP_SIGMOID: case FG_OP_TANH: case FG_OP_NEG:
      return K_ELEMWISE;
    case FG_OP_BADD_COL: case FG_OP_BMUL_COL: case FG_OP_BADD_ROW: case FG_OP_BMUL_ROW:
      return K_BROADCAST;
    case FG_OP_TRANSPOSE: case FG_OP_RESHAPE:
      return K_INJECTIVE;
    case FG_OP_ROWSUM: case FG_OP_ROWMAX:
      return K_COMM_REDUCE;
    case FG_OP_MATMUL_BF16:
      return K_OUT_EWISE_FUSABLE;
    case FG_OP_TUPLE:
      return K_TUPLE;
    case FG_OP_CONCAT:
      return K_INJECTIVE;
    default:
      return K_OPAQUE;
  }
}

namespace {

struct Fwd {
  int n = 0;
  std::vector<std::vector<int32_t>> succ;   // consumer nodes (deduplicated)
  std::vector<std::vector<int32_t>> ekind;  // pattern of each consumer edge
  std::vector<char> exits;                  // has an edge to the virtual exit
};

// Edge u -> v takes v's kind, except that a broadcast consumer reads an
// operand of its own output shape elementwise (the page's bias_add must let
// conv2d + bias_add + relu fuse in phase 0).
int edge_kind(const Graph& g, int32_t u, int32_t v) {
  const Node& nv = g.nodes[v];
  int k = op_kind(nv.op);
  if (k != K_BROADCAST) return k;
  const Value& out = g.values[nv.value];
  const Value& in = g.values[g.nodes[u].value];
  return in.same_shape(out) ? K_ELEMWISE : K_BROADCAST;
}

Fwd forward_graph(const Graph& g) {
  Fwd f;
  f.n = (int)g.nodes.size();
  f.succ.resize(f.n);
  f.ekind.resize(f.n);
  for (int v = 0; v < f.n; ++v) {
    for (int32_t a : g.nodes[v].args) {
      int u = g.values[a].node;
      if (u < 0) continue;
      auto& s = f.succ[u];
      if (std::find(s.begin(), s.end(), v) == s.end()) {
        s.push_back(v);
        f.ekind[u].push_back(edge_kind(g, u, v));
      }
    }
  }
  f.exits.resize(f.n);
  for (int u = 0; u < f.n; ++u)
    f.exits[u] = g.is_output[g.nodes[u].value] || f.succ[u].empty();
  return f;
}

// Immediate post-dominators in reverse topological order: the LCA of all
// consumers in the tree built so far.  While walking up, the path pattern
// (max edge kind over every path to the post-dominator) is accumulated from
// the patterns of the tree nodes passed: every path from a consumer to the
// LCA passes each post-dominator on the way, so the segments cover it.
void postdom(const Fwd& f, std::vector<int32_t>& parent, std::vector<int32_t>& depth,
             std::vector<int32_t>& ppat) {
  parent.assign(f.n, -1);
  depth.assign(f.n, 0);
  ppat.assign(f.n, 0);
  auto dep = [&](int x) { return x < 0 ? 0 : depth[x]; };
  for (int i = f.n - 1; i >= 0; --i) {
    if (f.exits[i]) {
      parent[i] = -1;
      depth[i] = 1;
      continue;
    }
    int lca = f.succ[i][0];
    int pat = f.ekind[i][0];
    for (size_t k = 1; k < f.succ[i].size(); ++k) {
      int a = lca, b = f.succ[i][k];
      pat = std::max(pat, f.ekind[i][k]);
      while (a != b) {
        if (dep(a) < dep(b)) std::swap(a, b);
        pat = std::max(pat, ppat[a]);
        a = parent[a];
      }
      lca = a;
    }
    parent[i] = lca;
    depth[i] = dep(lca) + 1;
    ppat[i] = pat;
  }
}

// Nodes strictly between src and sink on src -> sink paths (sink
// post-dominates src, so everything reachable from src short of sink is).
std::vector<int32_t> between(const Fwd& f, int src, int sink) {
  std::vector<int32_t> out, stack{src};
  std::vector<char> seen(f.n, 0);
  while (!stack.empty()) {
    int u = stack.back();
    stack.pop_back();
    for (int v : f.succ[u]) {
      if (v == sink || seen[v]) continue;
      seen[v] = 1;
      out.push_back(v);
      stack.push_back(v);
    }
  }
  return out;
}

struct UF {
  std::vector<int32_t> parent, pattern, size;
  explicit UF(const std::vector<int32_t>& kinds)
      : parent(kinds.size()), pattern(kinds), size(kinds.size(), 1) {
    for (size_t i = 0; i < kinds.size(); ++i) parent[i] = (int32_t)i;
  }
  int find(int x) const {
    while (parent[x] != x) x = parent[x];
    return x;
  }
};

}  // namespace

void partition(const Graph& g, const BuildOpts& o, std::vector<int32_t>& group_of,
               std::vector<int32_t>& ipdom) {
  Fwd f = forward_graph(g);
  std::vector<int32_t> depth, ppat;
  postdom(f, ipdom, depth, ppat);
  const int n = f.n;
  std::vector<int32_t> kinds(n);
  for (int i = 0; i < n; ++i) kinds[i] = op_kind(g.nodes[i].op);
  UF uf(kinds);

  auto check_path = [&](int src, int sink, auto cond) {
    for (int m : between(f, src, sink))
      if (!cond(uf.pattern[uf.find(m)], false)) return false;
    return (bool)cond(uf.pattern[uf.find(sink)], true);
  };

  for (int phase = 0; phase < 3; ++phase) {
    for (int i = 0; i < n; ++i) {
      int grp = uf.find(i);
      int gk = uf.pattern[grp];
      int p = ipdom[i];
      if (gk == K_OPAQUE || p < 0 || uf.find(p) == grp) continue;
      bool ok = false;
      if (gk == K_COMM_REDUCE) {
        // A reduction never starts a fusion, unless the reduce epilogue
        // option lets it take an elementwise tail on the reduced vector.
        if (o.allow_reduce_epilogue && ppat[i] == K_ELEMWISE) {
          ok = check_path(i, p, [](int k, bool) { return k == K_ELEMWISE; });
          const Value& red = g.values[g.nodes[i].value];
          std::vector<int32_t> path = between(f, i, p);
          path.push_back(p);
          for (int m : path)
            if (kinds[m] != K_ELEMWISE || !g.values[g.nodes[m].value].same_shape(red)) ok = false;
        }
      } else if (gk == K_OUT_EWISE_FUSABLE) {
        // Phase 0: fuse with an elementwise post-dominator when every node
        // up to it is broadcast or simpler.
        if (phase == 0 && ppat[i] == K_ELEMWISE)
          ok = check_path(i, p, [](int k, bool) { return k <= K_BROADCAST; });
      } else if (gk <= K_BROADCAST) {
        // Every phase: into an injective or reduce post-dominator; the sink
        // may already be an out-elementwise-fusable group.
        if (ppat[i] <= K_INJECTIVE || ppat[i] == K_COMM_REDUCE)
          ok = check_path(i, p, [](int k, bool is_sink) {
            if (!is_sink) return k <= K_INJECTIVE;
            return k <= K_INJECTIVE || k == K_COMM_REDUCE || k == K_OUT_EWISE_FUSABLE;
          });
      } else if (gk == K_INJECTIVE || gk == K_TUPLE) {
        // Phase 1: only along injective-or-simpler paths.
        if (phase == 1 && ppat[i] <= K_INJECTIVE)
          ok = check_path(i, p, [](int k, bool) { return k <= K_INJECTIVE; });
      }
      if (!ok && phase == 2) {
        // Phase 2: into an intermediate tuple that a later group absorbed.
        const int tg = uf.find(p);
        if (gk <= K_INJECTIVE && kinds[p] == K_TUPLE && uf.size[tg] > 1 && uf.pattern[tg] <= K_INJECTIVE)
          ok = check_path(i, p, [](int k, bool) { return k <= K_INJECTIVE; });
      }
      if (!ok) continue;

      std::vector<int32_t> touched = between(f, i, p);
      touched.push_back(i);
      touched.push_back(p);
      std::vector<int32_t> roots;
      for (int x : touched) {
        int r = uf.find(x);
        if (std::find(roots.begin(), roots.end(), r) == roots.end()) roots.push_back(r);
      }
      int64_t size = 0;
      for (int r : roots) size += uf.size[r];
      if (size > o.max_fused_ops) continue;
      // distinct values read from outside the merged group, plus its output
      std::vector<char> in(n, 0);
      for (int x = 0; x < n; ++x)
        if (std::find(roots.begin(), roots.end(), uf.find(x)) != roots.end()) in[x] = 1;
      std::vector<int32_t> ext;
      for (int x = 0; x < n; ++x) {
        if (!in[x]) continue;
        for (int32_t a : g.nodes[x].args) {
          int prod = g.values[a].node;
          if (prod >= 0 && in[prod]) continue;
          if (std::find(ext.begin(), ext.end(), a) == ext.end()) ext.push_back(a);
        }
      }
      if ((int64_t)ext.size() + 1 > o.max_args) continue;
      // CommitFuse: everything joins the post-dominator's group.
      int target = uf.find(p);
      for (int r : roots) {
        if (r == target) continue;
        uf.parent[r] = target;
        // an absorbed tuple counts as injective in the merged group
        const int a = uf.pattern[target] == K_TUPLE ? K_INJECTIVE : uf.pattern[target];
        const int b = uf.pattern[r] == K_TUPLE ? K_INJECTIVE : uf.pattern[r];
        uf.pattern[target] = std::max(a, b);
        uf.size[target] += uf.size[r];
      }
    }
  }
  group_of.assign(n, -1);
  std::vector<int32_t> sink(n, -1);
  for (int i = 0; i < n; ++i) {
    int r = uf.find(i);
    sink[r] = std::max(sink[r], i);
  }
  for (int i = 0; i < n; ++i) group_of[i] = sink[uf.find(i)];
}

}  // namespace fg
