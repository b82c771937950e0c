"""Post-dominator tree of the operator DAG.

TVM "Operator Fusion", FuseOps > Algorithm: step 1 builds a forward graph
whose nodes carry a pattern kind and consumer edges; step 2 finds each node's
immediate post-dominator -- the nearest downstream node that every future
path passes through -- as a least common ancestor on the DAG.  The diamond
shown there (one producer, three branches, one elementwise add) is the
motivating case.

Definition used here.  Nodes are operators (graph inputs are leaves, not
nodes).  A virtual EXIT node receives an edge from every node that is a graph
output or has no consumer.  d post-dominates n when d lies on every path
n -> EXIT; ipdom(n) is the nearest such d, reported as None when it is EXIT.
A graph output therefore always has ipdom None: its value leaves the graph.
"""
from __future__ import annotations

from .kinds import edge_kind, combine

NONE = -1


class ForwardGraph:
    """Node-indexed view of a GraphSpec: node i is the i-th operator."""

    def __init__(self, spec):
        self.spec = spec
        self.node_vid = [v.vid for v in spec.values if not v.is_input]
        self.vid_node = {vid: i for i, vid in enumerate(self.node_vid)}
        n = len(self.node_vid)
        self.n = n
        self.succ = [[] for _ in range(n)]       # consumer nodes, deduplicated
        for i, vid in enumerate(self.node_vid):
            for a in spec.values[vid].args:
                if a in self.vid_node:
                    p = self.vid_node[a]
                    if i not in self.succ[p]:
                        self.succ[p].append(i)
        outs = set(spec.outputs)
        self.to_exit = [(self.node_vid[i] in outs) or not self.succ[i] for i in range(n)]

    def kind(self, i):
        from .kinds import op_kind
        return op_kind(self.spec.values[self.node_vid[i]].op)

    def edge_kind(self, u, v):
        return edge_kind(self.spec, self.node_vid[u], self.node_vid[v])


def ipdom(fg: ForwardGraph):
    """Immediate post-dominators by LCA over consumers, in reverse topological
    order.  Returns (ipdom, depth) with depth(EXIT) = 0."""
    n = fg.n
    parent = [NONE] * n
    depth = [0] * n
    EXIT = n  # sentinel index for the walk

    def up(x):
        return parent[x] if parent[x] != NONE else EXIT

    def dep(x):
        return 0 if x == EXIT else depth[x]

    def lca(a, b):
        while a != b:
            if dep(a) < dep(b):
                a, b = b, a
            a = up(a)
        return a

    for i in range(n - 1, -1, -1):
        if fg.to_exit[i]:
            parent[i] = NONE
            depth[i] = 1
            continue
        anc = fg.succ[i][0]
        for c in fg.succ[i][1:]:
            anc = lca(anc, c)
        parent[i] = NONE if anc == EXIT else anc
        depth[i] = dep(anc) + 1
    return parent, depth


def nodes_between(fg: ForwardGraph, src: int, sink: int):
    """Nodes on some path src -> sink, excluding src and sink.  Valid when sink
    post-dominates src: every node reachable from src without passing sink
    lies on such a path."""
    seen, stack = set(), [src]
    while stack:
        u = stack.pop()
        for v in fg.succ[u]:
            if v != sink and v not in seen:
                seen.add(v)
                stack.append(v)
    return seen


def path_kind(fg: ForwardGraph, src: int, sink: int) -> int:
    """CombinePattern over every edge of every src -> sink path."""
    k = 0
    for u in [src] + sorted(nodes_between(fg, src, sink)):
        for v in fg.succ[u]:
            k = combine(k, fg.edge_kind(u, v))
    return k


def postdom_tree(spec):
    fg = ForwardGraph(spec)
    par, depth = ipdom(fg)
    pk = [path_kind(fg, i, par[i]) if par[i] != NONE else NONE for i in range(fg.n)]
    return fg, par, depth, pk
