"""Shared test helpers: brute-force graph checks, golden parsing, tolerances."""
from __future__ import annotations

import itertools
import os

import numpy as np

from workloads import GraphSpec

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Tolerances (per tensor): max_i |g_i - r_i| / max(|r_i|, rms(r)).
TOL_F32 = 1e-5
TOL_BF16 = 2e-2


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got)), "non-finite positions differ"
    assert np.array_equal(got[~fin], ref[~fin]), "infinities differ"
    if not fin.any():
        return 0.0
    r, g = ref[fin], got[fin]
    rms = np.sqrt(np.mean(r * r))
    den = np.maximum(np.abs(r), rms)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(g - r) / den))


# Operators whose float32 result is the correctly rounded value of their
# definition both on the GPU (the _rn intrinsics, never contracted into a
# fused multiply-add) and in the oracle (float64, then one rounding to float32:
# for +, -, * and / of float32 operands that double rounding cannot differ
# from a single one, since 53 >= 2 * 24 + 2), or that only move or select
# values.  A value computed through these alone must match bit for bit (the
# survey's reading R16: maxima and injective-only groups are bit-exact).
EXACT_OPS = frozenset({"add", "sub", "mul", "div", "scale", "addc", "relu", "neg", "badd_col", "bmul_col",
                       "badd_row", "bmul_row", "transpose", "reshape", "tuple", "concat", "rowmax",
                       "opaque_copy"})


def exact_value(spec, vid):
    """True when every operator that vid depends on is in EXACT_OPS."""
    seen, todo = set(), [vid]
    while todo:
        v = spec.values[todo.pop()]
        if v.is_input or v.vid in seen:
            continue
        seen.add(v.vid)
        if v.op not in EXACT_OPS:
            return False
        todo.extend(v.args)
    return True


def check_parity(spec, vid, got, ref, tol=TOL_F32):
    """Bit-exact for values computed by EXACT_OPS alone, else the per-tensor
    relative tolerance; returns the error (0 when bit-exact)."""
    got = np.asarray(got)
    if exact_value(spec, vid):
        np.testing.assert_array_equal(got, np.asarray(ref), err_msg=f"value {vid} ({spec.values[vid].op})")
        return 0.0
    e = rel_err(got, ref)
    assert e <= tol, (vid, spec.values[vid].op, e)
    return e


def read_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.rstrip("\n") for ln in f if ln.strip() and not ln.startswith("#")]


def graph_from_golden(name):
    g = GraphSpec(name)
    expect = {}
    for ln in read_golden(name):
        tok = ln.split()
        if tok[1] == "input":
            g.input(tuple(int(s) for s in tok[2].split(",")))
        elif tok[1] == "op":
            args = [int(a) for a in tok[3].split(",")]
            attrs = () if tok[4] == "-" else tuple(float(a) for a in tok[4].split(","))
            g.op(tok[2], args, attrs)
        elif tok[0] == "output":
            g.mark_output(int(tok[1]))
        else:
            expect[tok[0]] = [int(a) for a in tok[1].split(",")]
    return g, expect


# -- brute force on node DAGs -------------------------------------------------

def node_succ(spec):
    node_vid = [v.vid for v in spec.values if not v.is_input]
    vid_node = {v: i for i, v in enumerate(node_vid)}
    succ = [set() for _ in node_vid]
    for i, vid in enumerate(node_vid):
        for a in spec.values[vid].args:
            if a in vid_node:
                succ[vid_node[a]].add(i)
    outs = set(spec.outputs)
    exits = [(node_vid[i] in outs) or not succ[i] for i in range(len(node_vid))]
    return node_vid, [sorted(s) for s in succ], exits


def all_paths_to_exit(succ, exits, n):
    """Every path from node n to the virtual EXIT, as node lists (n excluded)."""
    out = []

    def walk(u, acc):
        if exits[u]:
            out.append(acc + ["EXIT"])
        for v in succ[u]:
            walk(v, acc + [v])
    walk(n, [])
    return out


def brute_ipdom(succ, exits, n):
    paths = all_paths_to_exit(succ, exits, n)
    common = set(paths[0])
    for p in paths[1:]:
        common &= set(p)
    for x in paths[0]:          # common nodes appear in the same order on every path
        if x in common:
            return -1 if x == "EXIT" else x
    raise AssertionError("EXIT is always common")


def brute_paths_between(succ, a, b):
    out = []

    def walk(u, acc):
        if u == b:
            out.append(acc)
            return
        for v in succ[u]:
            walk(v, acc + [v])
    walk(a, [a])
    return out


def small_dags(max_nodes, max_preds=3, seed=None, count=None):
    """Yield (n, preds) for every DAG on n <= max_nodes nodes where node j
    reads up to max_preds earlier nodes (exhaustive), or `count` random ones."""
    if seed is None:
        for n in range(1, max_nodes + 1):
            choices = []
            for j in range(n):
                subs = [()]
                for k in range(1, min(max_preds, j) + 1):
                    subs += list(itertools.combinations(range(j), k))
                choices.append(subs)
            for preds in itertools.product(*choices):
                yield n, preds
    else:
        rng = np.random.default_rng(seed)
        for _ in range(count):
            n = int(rng.integers(2, max_nodes + 1))
            preds = []
            for j in range(n):
                k = int(rng.integers(0, min(max_preds, j) + 1))
                preds.append(tuple(sorted(rng.choice(j, size=k, replace=False).tolist())) if k else ())
            yield n, tuple(preds)


UNARY = ("relu", "transpose", "rowsum", "opaque_copy", "exp")
NARY = ("add", "mul", "badd_col")


def dag_to_spec(n, preds, op_choice=None, outputs=()):
    """A GraphSpec over square [4,4] values realising the node DAG `preds`;
    nodes with no predecessor read a fresh input.  `op_choice[j]` picks the
    operator among those of the right arity."""
    g = GraphSpec("dag")
    vid_of = []
    for j in range(n):
        args = [vid_of[p] for p in preds[j]]
        if not args:
            args = [g.input((4, 4))]
        k = 0 if op_choice is None else op_choice[j]
        if len(args) == 1:
            op = UNARY[k % len(UNARY)]
            if len(g.values[args[0]].shape) == 1 and op in ("transpose", "rowsum"):
                op = "relu"
        elif len(args) == 2:
            op = NARY[k % len(NARY)]
        else:
            op = "add"
        vid_of.append(g.op(op, args))
    for o in outputs:
        g.mark_output(vid_of[o])
    return g


def tuple_dag(seed):
    """Random branches (elementwise, with inputs of their own, or opaque
    copies) joined by a tuple, usually concatenated, then a short tail."""
    r = np.random.default_rng(seed)
    g = GraphSpec("tuples")
    C = int(r.choice([8, 12, 16]))
    fields = []
    for _ in range(int(r.integers(2, 5))):
        rows = int(r.choice([4, 8, 12, 16]))
        v = g.input((rows, C))
        for _ in range(int(r.integers(0, 3))):
            k = int(r.integers(0, 4))
            if k == 0:
                v = g.op("relu", (v,))
            elif k == 1:
                v = g.op("scale", (v,), (0.5,))
            elif k == 2:
                v = g.op("add", (v, g.input((rows, C))))
            else:
                v = g.op("opaque_copy", (v,))
        fields.append(v)
    t = g.op("tuple", tuple(fields))
    if r.random() < 0.8:
        t = g.op("concat", (t,))
    tail = int(r.integers(0, 4))
    for _ in range(tail):
        k = int(r.integers(0, 3))
        t = g.op("exp", (t,)) if k == 0 else g.op("transpose", (t,)) if k == 1 else g.op("rowsum", (t,))
        if len(g.values[t].shape) == 1:
            break
    g.mark_output(t)
    if r.random() < 0.3:
        g.mark_output(fields[0]) if not g.values[fields[0]].is_input else None
    return g
