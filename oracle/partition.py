"""FuseOps grouping: CheckPath / CommitFuse with union-find, phases 0, 1 and 2.

TVM "Operator Fusion", FuseOps > Algorithm (step 3) and Fusion rules:

* every node, in topological order, tries to fuse with its immediate
  post-dominator; CheckPath tests every node on every path between them,
  CommitFuse unions those nodes' groups (union-find);
* phase 0: an out-elementwise-fusable group (matmul) fuses with an
  elementwise post-dominator when every node up to it is broadcast or
  simpler; two such groups never fuse;
* elementwise/broadcast groups fuse in every phase into an injective or
  reduce post-dominator; intermediate nodes may be injective or simpler and
  the sink may also already be an out-elementwise-fusable group;
* phase 1: injective groups fuse when every path is injective or simpler;
* a reduction never starts a fusion, an opaque node is a barrier, and a group
  holds at most kMaxFusedOps (256) nodes and a bounded number of arguments.

Readings where the page is silent (each mirrored by the C++ partitioner):
* topological order = creation order;
* the "elementwise post-dominator" of phase 0 is the path pattern (edge kinds,
  see ``kinds.edge_kind``), not the node kind;
* the argument limit is ``max_args`` (default 64) counting distinct values
  read from outside the merged group plus its one output;
* an elementwise producer never joins a matmul group through the matmul's own
  operand: that edge has the matmul's kind, which the path test rejects;
* a tuple fuses like an injective op in phase 1 (every path to its
  post-dominator injective or simpler); once merged into a group with other
  operators it counts as injective in that group's pattern, so absorbing a
  tuple does not make a concatenation's group more complex;
* phase 2: an operator whose group is injective or simpler and whose
  immediate post-dominator is a tuple already absorbed by a later group (the
  tuple's group holds more than the tuple and is injective or simpler) fuses
  into that group when every node between them is injective or simpler;
* ``allow_reduce_epilogue`` (off by default) lets a reduce group absorb its
  post-dominator when every node on the way is elementwise on the reduced
  shape, a DisCo-style fusion of an op with its predecessor (DisCo Sec. 3.2,
  strategy (i)) that the TVM rules alone do not allow.
"""
from __future__ import annotations

from dataclasses import dataclass

from .kinds import (K_ELEMWISE, K_BROADCAST, K_INJECTIVE, K_COMM_REDUCE,
                    K_OUT_EWISE_FUSABLE, K_TUPLE, K_OPAQUE, combine)
from .postdom import postdom_tree, nodes_between, NONE


@dataclass
class Options:
    max_fused_ops: int = 256
    max_args: int = 64
    allow_reduce_epilogue: bool = False


class UnionFind:
    def __init__(self, n, kinds):
        self.parent = list(range(n))
        self.pattern = list(kinds)
        self.size = [1] * n

    def find(self, x):
        while self.parent[x] != x:
            x = self.parent[x]
        return x

    def union_into(self, child_root, root):
        if child_root == root:
            return
        self.parent[child_root] = root
        # an absorbed tuple counts as injective in the merged group
        a, b = self.pattern[root], self.pattern[child_root]
        a = K_INJECTIVE if a == K_TUPLE else a
        b = K_INJECTIVE if b == K_TUPLE else b
        self.pattern[root] = combine(a, b)
        self.size[root] += self.size[child_root]


def _merged_nodes(uf, fg, touched):
    roots = {uf.find(x) for x in touched}
    return [i for i in range(fg.n) if uf.find(i) in roots]


def _num_args(fg, nodes):
    """Distinct values read by `nodes` that are produced outside them, + 1 output."""
    spec = fg.spec
    inside = {fg.node_vid[i] for i in nodes}
    ext = set()
    for i in nodes:
        for a in spec.values[fg.node_vid[i]].args:
            if a not in inside:
                ext.add(a)
    return len(ext) + 1


def partition(spec, opts: Options | None = None):
    """Return (group_of, ipdom) with group_of[node] = the group's largest node
    index (its sink) and ipdom[node] = immediate post-dominator or -1."""
    opts = opts or Options()
    fg, par, _depth, pk = postdom_tree(spec)
    n = fg.n
    kinds = [fg.kind(i) for i in range(n)]
    uf = UnionFind(n, kinds)

    def check_path(src, sink, cond):
        for m in nodes_between(fg, src, sink):
            if not cond(uf.pattern[uf.find(m)], False):
                return False
        return cond(uf.pattern[uf.find(sink)], True)

    for phase in (0, 1, 2):
        for i in range(n):
            g = uf.find(i)
            gk = uf.pattern[g]
            p = par[i]
            if gk == K_OPAQUE or p == NONE or uf.find(p) == g:
                continue
            ok = False
            if gk == K_COMM_REDUCE:
                # a reduction never initiates fusion (optional epilogue below)
                if opts.allow_reduce_epilogue and pk[i] == K_ELEMWISE:
                    red_shape = spec.values[fg.node_vid[i]].shape
                    path = list(nodes_between(fg, i, p)) + [p]
                    ok = (check_path(i, p, lambda k, s: k == K_ELEMWISE) and
                          all(kinds[m] == K_ELEMWISE and
                              spec.values[fg.node_vid[m]].shape == red_shape for m in path))
            elif gk == K_OUT_EWISE_FUSABLE:
                if phase == 0 and pk[i] == K_ELEMWISE:
                    ok = check_path(i, p, lambda k, s: k <= K_BROADCAST)
            elif gk <= K_BROADCAST:
                if pk[i] <= K_INJECTIVE or pk[i] == K_COMM_REDUCE:
                    def cond(k, is_sink):
                        if not is_sink:
                            return k <= K_INJECTIVE
                        return k <= K_INJECTIVE or k in (K_COMM_REDUCE, K_OUT_EWISE_FUSABLE)
                    ok = check_path(i, p, cond)
            elif gk in (K_INJECTIVE, K_TUPLE):
                if phase == 1 and pk[i] <= K_INJECTIVE:
                    ok = check_path(i, p, lambda k, s: k <= K_INJECTIVE)
            if not ok and phase == 2:
                # into an intermediate tuple that a later group has absorbed
                tg = uf.find(p)
                if (gk <= K_INJECTIVE and kinds[p] == K_TUPLE and uf.size[tg] > 1
                        and uf.pattern[tg] <= K_INJECTIVE):
                    ok = check_path(i, p, lambda k, s: k <= K_INJECTIVE)
            if not ok:
                continue
            # size and argument limits on the merged group
            touched = [i, p] + list(nodes_between(fg, i, p))
            merged = _merged_nodes(uf, fg, touched)
            if len(merged) > opts.max_fused_ops:
                continue
            if _num_args(fg, merged) > opts.max_args:
                continue
            # CommitFuse
            target = uf.find(p)
            for r in {uf.find(x) for x in touched}:
                uf.union_into(r, target)
    group_of = [0] * n
    sink = {}
    for i in range(n):
        r = uf.find(i)
        sink[r] = max(sink.get(r, -1), i)
    for i in range(n):
        group_of[i] = sink[uf.find(i)]
    return group_of, par


def groups(spec, opts: Options | None = None):
    """Groups as {sink node: sorted node list}, plus ipdom."""
    group_of, par = partition(spec, opts)
    out = {}
    for i, gsink in enumerate(group_of):
        out.setdefault(gsink, []).append(i)
    return out, par


def group_io(spec, nodes):
    """Leaves (values read from outside, in first-use order), the output value
    and the algorithmic bytes (each leaf read once, the output written once)."""
    node_vid = [v.vid for v in spec.values if not v.is_input]
    inside = [node_vid[i] for i in sorted(nodes)]
    inside_set = set(inside)
    leaves = []
    for vid in inside:
        for a in spec.values[vid].args:
            if a not in inside_set and a not in leaves:
                leaves.append(a)
    out = inside[-1]

    def nbytes(vid):
        v = spec.values[vid]
        n = 1
        for s in v.shape:
            n *= s
        return n * (2 if v.dtype == "bf16" else 4)
    alg = sum(nbytes(v) for v in leaves) + nbytes(out)
    return leaves, out, alg
