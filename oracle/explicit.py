"""Explicit fusion moves on a partition of a graph's operators (test
infrastructure: only tests, the smoke check and the bench's CPU legs use
this module).

DisCo, Introduction: an operator is fused with one of its predecessors (an
operator whose output it reads).  When that predecessor has other
successors, *non-duplicate* fusion folds it into the fused operator, so its
output reaches its other readers only when the fused operator completes;
*duplicate* fusion fuses it and also recomputes it outside the fused
operator.  DisCo, Strategy Maker, optimisation methods (i) and (ii) are these
two moves; the search that picks them is out of scope here.

Readings where the pages are silent:

* a group must stay convex: no path may leave it and come back, otherwise
  the groups could not run one after another;
* duplicate fusion appends a copy of the predecessor (next node and value
  ids) that joins the reader's group and feeds it; the original keeps its
  group and its other readers; when nothing else reads the predecessor both
  moves merge the two groups;
* a group is labelled by its smallest node id; groups run in the order of
  their dependencies, smallest label first among those ready;
* a group's outputs: its sink (the last member whose value no member
  reads), then every other member whose value an outside operator reads, the
  caller receives (a graph output), or nobody reads.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass, field

from oracle import partition as OP
from oracle import execute as OE


@dataclass
class State:
    ops: list                      # per node: [op, args, attrs, out vid]
    label: list                    # per node: group label
    clone_of: list                 # per node: copied node or -1
    n_values: int                  # value ids in use
    outputs: list = field(default_factory=list)


def initial(spec, from_fuseops=True, opts=None):
    ops = [[v.op, tuple(v.args), tuple(v.attrs), v.vid] for v in spec.ops]
    n = len(ops)
    if from_fuseops:
        group_of, _ = OP.partition(spec, opts)
        first = {}
        for i, gs in enumerate(group_of):
            first.setdefault(gs, i)
        label = [first[group_of[i]] for i in range(n)]
    else:
        label = list(range(n))
    return State(ops, label, [-1] * n, len(spec.values), list(spec.outputs))


def _producer(st):
    return {o[3]: i for i, o in enumerate(st.ops)}


def members(st, lab):
    return [i for i, l in enumerate(st.label) if l == lab]


def is_convex(st, nodes):
    """No path from a member through a non-member back to a member."""
    inside = set(nodes)
    prod = _producer(st)
    readers = {}
    for i, o in enumerate(st.ops):
        for a in o[1]:
            if a in prod:
                readers.setdefault(prod[a], set()).add(i)
    frontier = [y for x in inside for y in readers.get(x, ()) if y not in inside]
    seen = set(frontier)
    while frontier:
        x = frontier.pop()
        for y in readers.get(x, ()):
            if y in inside:
                return False
            if y not in seen:
                seen.add(y)
                frontier.append(y)
    return True


class NotConvex(Exception):
    pass


def fuse(st, node, pred, duplicate=False):
    """The state after fusing operator `node` with its predecessor `pred`."""
    pv = st.ops[pred][3]
    if pv not in st.ops[node][1]:
        raise ValueError("not a predecessor")
    if st.label[node] == st.label[pred]:
        raise ValueError("already in one group")
    shared = pv in st.outputs or any(pv in o[1] for i, o in enumerate(st.ops) if i != node)
    s = copy.deepcopy(st)
    if duplicate and shared:
        op, args, attrs, _ = s.ops[pred]
        cv = s.n_values
        s.n_values += 1
        s.ops.append([op, args, attrs, cv])
        s.ops[node][1] = tuple(cv if a == pv else a for a in s.ops[node][1])
        s.label.append(s.label[node])
        s.clone_of.append(st.clone_of[pred] if st.clone_of[pred] >= 0 else pred)
        if not is_convex(s, members(s, s.label[node])):
            raise NotConvex()
        return s
    la, lb = st.label[node], st.label[pred]
    merged = members(st, la) + members(st, lb)
    if not is_convex(st, merged):
        raise NotConvex()
    nl = min(la, lb)
    s.label = [nl if l in (la, lb) else l for l in s.label]
    return s


def groups(st):
    """Node lists of the groups, each after the groups whose outputs it reads."""
    labels = sorted(set(st.label))
    prod = _producer(st)
    deps = {l: set() for l in labels}
    for i, o in enumerate(st.ops):
        for a in o[1]:
            if a in prod and st.label[prod[a]] != st.label[i]:
                deps[st.label[i]].add(st.label[prod[a]])
    done, order = set(), []
    while len(order) < len(labels):
        ready = [l for l in labels if l not in done and deps[l] <= done]
        l = min(ready)
        done.add(l)
        order.append(members(st, l))
    return order


def group_outputs(st, nodes):
    """[sink value, extra output values...] of a group."""
    inside = set(nodes)
    read_in = {a for i in nodes for a in st.ops[i][1]}
    read_out = {a for i, o in enumerate(st.ops) if i not in inside for a in o[1]}
    sink = max(i for i in nodes if st.ops[i][3] not in read_in)
    sv = st.ops[sink][3]
    extra = [st.ops[i][3] for i in sorted(nodes)
             if st.ops[i][3] != sv and (st.ops[i][3] in read_out or st.ops[i][3] in st.outputs
                                        or st.ops[i][3] not in read_in)]
    return [sv] + extra


def run(st, inputs):
    """Every operator of the transformed graph, group by group (one operator
    at a time inside a group, in dependency order); returns every value."""
    env = dict(inputs)
    for nodes in groups(st):
        pending = sorted(nodes)
        while pending:
            for i in pending:
                op, args, attrs, out = st.ops[i]
                if all(a in env for a in args):
                    env[out] = OE.apply_op(op, [env[a] for a in args], attrs)
                    pending.remove(i)
                    break
            else:
                raise AssertionError("group without a runnable operator")
    return env
