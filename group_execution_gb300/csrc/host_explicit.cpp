// Explicit fusion: a partition of a graph's operators changed one move at a
// time (DisCo, Introduction: an operator is fused with one of the
// predecessors whose output it reads; when that predecessor has other
// successors, non-duplicate fusion folds it into the fused operator, whose
// completion its other readers then wait for, while duplicate fusion also
// recomputes it outside; Strategy Maker, optimisation methods (i) and (ii)).
//
// A move is accepted only if the merged group stays convex (no path leaves it
// and comes back, else the groups could not run one after another) and the
// caller's check (the group compiles into one kernel) passes.
#include <algorithm>
#include <deque>
#include <queue>

#include "host.h"

namespace fg {

namespace {

[[noreturn]] void fail(fg_status st, const std::string& msg) { throw CompileError{st, msg}; }

std::vector<std::vector<int32_t>> consumers_of(const Graph& g) {
  std::vector<std::vector<int32_t>> c(g.values.size());
  for (size_t x = 0; x < g.nodes.size(); ++x)
    for (int32_t a : g.nodes[x].args)
      if (c[a].empty() || c[a].back() != (int32_t)x) c[a].push_back((int32_t)x);
  return c;
}

// No path from a member through a non-member back to a member.
bool convex(const Graph& g, const std::vector<char>& in) {
  const auto cons = consumers_of(g);
  std::vector<char> seen(g.nodes.size(), 0);
  std::deque<int32_t> q;
  for (size_t x = 0; x < g.nodes.size(); ++x)
    if (in[x])
      for (int32_t y : cons[g.nodes[x].value])
        if (!in[y] && !seen[y]) {
          seen[y] = 1;
          q.push_back(y);
        }
  while (!q.empty()) {
    const int32_t x = q.front();
    q.pop_front();
    for (int32_t y : cons[g.nodes[x].value]) {
      if (in[y]) return false;
      if (!seen[y]) {
        seen[y] = 1;
        q.push_back(y);
      }
    }
  }
  return true;
}

std::vector<int32_t> members(const Partition& P, int32_t label) {
  std::vector<int32_t> m;
  for (size_t x = 0; x < P.label.size(); ++x)
    if (P.label[x] == label) m.push_back((int32_t)x);
  return m;
}

void check_group(const Partition& P, const std::vector<int32_t>& nodes, const GroupCheck& check) {
  std::vector<char> in(P.g.nodes.size(), 0);
  for (int32_t x : nodes) in[x] = 1;
  if (!convex(P.g, in)) fail(FG_EUNSUPPORTED, "the fused group would not be convex (a path leaves it and returns)");
  if ((int)nodes.size() > P.max_fused_ops) fail(FG_EUNSUPPORTED, "the fused group exceeds max_fused_ops");
  check(P.g, nodes);
}

}  // namespace

Partition singleton_partition(const Graph& g, const BuildOpts& o) {
  Partition P;
  P.g = g;
  P.max_fused_ops = o.max_fused_ops;
  for (size_t x = 0; x < g.nodes.size(); ++x) {
    P.label.push_back((int32_t)x);
    P.clone_of.push_back(-1);
  }
  return P;
}

void fuse_move(Partition& P, int32_t node, int32_t pred, bool duplicate, const GroupCheck& check) {
  const int32_t n = (int32_t)P.g.nodes.size();
  if (node < 0 || node >= n || pred < 0 || pred >= n) fail(FG_EINVAL, "node id out of range");
  const int32_t pv = P.g.nodes[pred].value;
  const auto& args = P.g.nodes[node].args;
  if (std::find(args.begin(), args.end(), pv) == args.end())
    fail(FG_EINVAL, "the predecessor's output is not an operand of the node");
  if (P.label[node] == P.label[pred]) fail(FG_EINVAL, "the two operators are already in one group");
  // does anything but `node` read the predecessor's output?
  bool shared = P.g.is_output[pv] != 0;
  for (int32_t x = 0; x < n && !shared; ++x)
    if (x != node) {
      const auto& a = P.g.nodes[x].args;
      shared = std::find(a.begin(), a.end(), pv) != a.end();
    }
  if (duplicate && shared) {
    // a copy of the predecessor joins the node's group and feeds the node;
    // the original keeps serving its other readers
    Partition Q = P;
    Node copy = Q.g.nodes[pred];
    Value cv = Q.g.values[pv];
    cv.node = n;
    cv.is_input = false;
    copy.value = (int32_t)Q.g.values.size();
    Q.g.values.push_back(cv);
    Q.g.is_output.push_back(0);
    Q.g.nodes.push_back(copy);
    for (int32_t& a : Q.g.nodes[node].args)
      if (a == pv) a = copy.value;
    Q.label.push_back(Q.label[node]);
    Q.clone_of.push_back(P.clone_of[pred] >= 0 ? P.clone_of[pred] : pred);
    check_group(Q, members(Q, Q.label[node]), check);
    P = std::move(Q);
    return;
  }
  // non-duplicate fusion (for a predecessor nothing else reads, both kinds
  // are the same move): the two groups merge
  const int32_t la = P.label[node], lb = P.label[pred];
  std::vector<int32_t> m = members(P, la), mb = members(P, lb);
  m.insert(m.end(), mb.begin(), mb.end());
  check_group(P, m, check);
  const int32_t nl = std::min(la, lb);
  for (int32_t& l : P.label)
    if (l == la || l == lb) l = nl;
}

std::vector<std::vector<int32_t>> partition_groups(const Partition& P) {
  // groups by label, ordered so that every group runs after the groups whose
  // outputs it reads (Kahn's algorithm, smallest label first)
  std::vector<int32_t> labels;
  for (int32_t l : P.label)
    if (std::find(labels.begin(), labels.end(), l) == labels.end()) labels.push_back(l);
  std::sort(labels.begin(), labels.end());
  std::vector<int32_t> gi(P.g.nodes.size());
  for (size_t x = 0; x < P.label.size(); ++x)
    gi[x] = (int32_t)(std::lower_bound(labels.begin(), labels.end(), P.label[x]) - labels.begin());
  const int G = (int)labels.size();
  std::vector<std::vector<int32_t>> succ(G);
  std::vector<int> indeg(G, 0);
  for (size_t x = 0; x < P.g.nodes.size(); ++x)
    for (int32_t a : P.g.nodes[x].args) {
      const int32_t prod = P.g.values[a].node;
      if (prod < 0 || gi[prod] == gi[x]) continue;
      auto& s = succ[gi[prod]];
      if (std::find(s.begin(), s.end(), gi[x]) == s.end()) {
        s.push_back(gi[x]);
        ++indeg[gi[x]];
      }
    }
  std::priority_queue<int, std::vector<int>, std::greater<int>> ready;
  for (int k = 0; k < G; ++k)
    if (!indeg[k]) ready.push(k);
  std::vector<std::vector<int32_t>> out;
  while (!ready.empty()) {
    const int k = ready.top();
    ready.pop();
    out.push_back(members(P, labels[k]));
    for (int32_t t : succ[k])
      if (--indeg[t] == 0) ready.push(t);
  }
  if ((int)out.size() != G) fail(FG_EUNSUPPORTED, "internal: groups form a cycle");
  return out;
}

// Pattern-based grouping (TVM "Operator Fusion", FuseOpsByPattern): anchors
// in node order, patterns in priority order at each anchor; a chain's next
// operator is the smallest-numbered untaken reader of the previous output
// with the pattern's operator; a match must be convex, pass the private
// check when asked (no intermediate result read outside it or returned) and
// run as one kernel; everything else stays alone.
Partition pattern_partition(const Graph& g, const BuildOpts& o, const std::vector<ChainPattern>& pats,
                            const GroupCheck& check, std::vector<int32_t>& match_of) {
  Partition P = singleton_partition(g, o);
  const int n = (int)g.nodes.size();
  const auto cons = consumers_of(g);
  std::vector<char> taken(n, 0);
  match_of.assign(n, -1);
  for (int anchor = 0; anchor < n; ++anchor) {
    if (taken[anchor]) continue;
    for (size_t k = 0; k < pats.size(); ++k) {
      const ChainPattern& pt = pats[k];
      if (pt.ops.empty() || g.nodes[anchor].op != pt.ops[0]) continue;
      std::vector<int32_t> chain{anchor};
      for (size_t j = 1; j < pt.ops.size() && !chain.empty(); ++j) {
        int next = -1;
        for (int32_t r : cons[g.nodes[chain.back()].value])   // readers in node order
          if (!taken[r] && g.nodes[r].op == pt.ops[j] && std::find(chain.begin(), chain.end(), r) == chain.end()) {
            next = r;
            break;
          }
        if (next < 0) chain.clear();
        else chain.push_back(next);
      }
      if (chain.empty()) continue;
      std::vector<char> in(n, 0);
      for (int32_t x : chain) in[x] = 1;
      if (!convex(g, in)) continue;
      if (pt.private_intermediates) {
        bool ok = true;
        for (size_t j = 0; j + 1 < chain.size() && ok; ++j) {
          const int32_t v = g.nodes[chain[j]].value;
          if (g.is_output[v]) ok = false;
          for (int32_t r : cons[v])
            if (!in[r]) ok = false;
        }
        if (!ok) continue;
      }
      if (chain.size() > 1) {
        try {
          check(g, chain);
        } catch (const CompileError&) {
          continue;
        }
      }
      const int32_t lab = *std::min_element(chain.begin(), chain.end());
      for (int32_t x : chain) {
        taken[x] = 1;
        match_of[x] = (int32_t)k;
        P.label[x] = lab;
      }
      break;
    }
  }
  return P;
}

}  // namespace fg
