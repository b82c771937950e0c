"""Pins for the oracle's post-dominator tree (TVM "Operator Fusion", FuseOps >
Algorithm, steps 1-2): the LCA construction must agree exactly with the plain
definition, evaluated by enumerating every path to the virtual exit."""
import numpy as np

from oracle import postdom, kinds
from tests._helpers import (small_dags, dag_to_spec, node_succ, brute_ipdom,
                            brute_paths_between)
import workloads as W


def _check(spec):
    fg, par, _, pk = postdom.postdom_tree(spec)
    _, succ, exits = node_succ(spec)
    for i in range(fg.n):
        assert par[i] == brute_ipdom(succ, exits, i), (i, par)
        if par[i] >= 0:
            k = 0
            for path in brute_paths_between(succ, i, par[i]):
                for u, v in zip(path, path[1:]):
                    k = max(k, fg.edge_kind(u, v))
            assert pk[i] == k


def test_ipdom_exhaustive_small_dags():
    """Every DAG on up to 5 nodes (<= 3 operands per node), with and without
    an interior node marked as a graph output."""
    cnt = 0
    for n, preds in small_dags(5):
        _check(dag_to_spec(n, preds))
        if n >= 3:
            _check(dag_to_spec(n, preds, outputs=(n // 2,)))
        cnt += 1
    assert cnt > 900


def test_ipdom_random_dags_up_to_7_nodes():
    rng = np.random.default_rng(7)
    for n, preds in small_dags(7, seed=11, count=2500):
        ops = rng.integers(0, 5, size=n)
        outs = tuple(rng.choice(n, size=int(rng.integers(0, 2)), replace=False).tolist())
        _check(dag_to_spec(n, preds, ops, outs))


def test_diamond_from_the_page():
    """One producer, three branches, reconverging at an elementwise add: the
    add is the producer's immediate post-dominator."""
    g = W.diamond(16, 8)
    fg, par, _, pk = postdom.postdom_tree(g)
    # nodes: 0 badd_col (P), 1 relu, 2 scale, 3 exp, 4 mul, 5 add, 6 transpose
    assert par[0] == 5
    assert par[1] == 5 and par[3] == 5 and par[4] == 5 and par[2] == 3
    assert par[5] == 6 and par[6] == -1
    assert pk[0] == kinds.K_ELEMWISE
    assert pk[5] == kinds.K_INJECTIVE


def test_graph_output_is_always_a_root():
    g = W.GraphSpec()
    x = g.input((4, 4))
    a = g.op("relu", (x,))
    b = g.op("exp", (a,))
    g.mark_output(a)
    g.mark_output(b)
    _, par, _, _ = postdom.postdom_tree(g)
    assert par == [-1, -1]


def test_edge_kinds_of_bias_add():
    """bias_add is broadcast (TVM, Pattern Classification): its vector operand
    is a broadcast edge, its same-shape operand an elementwise one."""
    g = W.GraphSpec()
    x = g.input((4, 8))
    v = g.input((8,))
    m = g.op("relu", (x,))
    vv = g.op("exp", (v,))
    b = g.op("badd_col", (m, vv))
    assert kinds.edge_kind(g, m, b) == kinds.K_ELEMWISE
    assert kinds.edge_kind(g, vv, b) == kinds.K_BROADCAST


def test_pattern_kind_values_from_the_page():
    assert (kinds.K_ELEMWISE, kinds.K_BROADCAST, kinds.K_INJECTIVE, kinds.K_COMM_REDUCE,
            kinds.K_OUT_EWISE_FUSABLE, kinds.K_TUPLE, kinds.K_OPAQUE) == (0, 1, 2, 3, 4, 7, 8)
    assert kinds.op_kind("transpose") == kinds.K_INJECTIVE      # not broadcast
    assert kinds.op_kind("badd_col") == kinds.K_BROADCAST
    assert kinds.op_kind("matmul_bf16") == kinds.K_OUT_EWISE_FUSABLE
    assert kinds.combine(kinds.K_BROADCAST, kinds.K_INJECTIVE) == kinds.K_INJECTIVE
