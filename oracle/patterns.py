"""Pattern-based grouping (test infrastructure: only tests, the smoke check
and the bench's CPU legs use this module).

TVM "Operator Fusion", FuseOpsByPattern: the caller names which operator
combinations form a group (a pattern such as matmul(x, w) + bias); patterns
are given in priority order and when a subgraph matches several the first
pattern wins; a check may reject a match, for instance when an intermediate
result is used outside the group.

Readings where the page is silent: a pattern is a chain of operators, each
reading the previous one's output as any of its operands (the other operands
are wildcards); anchors are tried in node order, and at each anchor the
patterns in priority order; along the chain the next operator is the
smallest-numbered reader of the previous output with the pattern's operator;
an operator already in a match cannot join another; a match must be convex
(no path leaves it and comes back) to run as one group; the built-in check
(`private`) rejects a match whose intermediate results are read outside it
or returned to the caller; operators outside every match stay alone.
"""
from __future__ import annotations


def match(spec, patterns):
    """patterns: list of (name, [op names], private).  Returns (groups,
    match_of): groups as sorted node lists (matches and singletons, by first
    node), match_of[node] = index of the matching pattern or -1."""
    node_of = spec.node_of_value()
    ops = spec.ops
    readers = {}
    for i, v in enumerate(ops):
        for a in v.args:
            if a in node_of:
                readers.setdefault(node_of[a], [])
                if i not in readers[node_of[a]]:
                    readers[node_of[a]].append(i)
    taken = [False] * len(ops)
    match_of = [-1] * len(ops)
    matches = []
    for anchor in range(len(ops)):
        if taken[anchor]:
            continue
        for k, (_name, chain, private) in enumerate(patterns):
            if ops[anchor].op != chain[0]:
                continue
            nodes = [anchor]
            for want in chain[1:]:
                nxt = [r for r in sorted(readers.get(nodes[-1], [])) if ops[r].op == want and not taken[r]]
                if not nxt:
                    nodes = None
                    break
                nodes.append(nxt[0])
            if nodes is None:
                continue
            if not _convex(readers, set(nodes)):
                continue
            if private:
                inside = set(nodes)
                bad = False
                for x in nodes[:-1]:
                    vid = ops[x].vid
                    if vid in spec.outputs or any(r not in inside for r in readers.get(x, [])):
                        bad = True
                if bad:
                    continue
            for x in nodes:
                taken[x] = True
                match_of[x] = k
            matches.append(sorted(nodes))
            break
    groups = matches + [[i] for i in range(len(ops)) if not taken[i]]
    groups.sort(key=lambda g: g[0])
    return groups, match_of


def _convex(readers, inside):
    """No path from a member through a non-member back to a member."""
    frontier = [y for x in inside for y in readers.get(x, []) if y not in inside]
    seen = set(frontier)
    while frontier:
        x = frontier.pop()
        for y in readers.get(x, []):
            if y in inside:
                return False
            if y not in seen:
                seen.add(y)
                frontier.append(y)
    return True
