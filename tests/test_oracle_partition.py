"""Pins for the oracle's FuseOps grouping: the worked example and the rules
stated on the TVM "Operator Fusion" page (FuseOps > Example, Fusion rules and
the constraints under them), plus invariants checked by brute force."""
import numpy as np
import pytest

from oracle import partition as P, kinds
from tests._helpers import (graph_from_golden, small_dags, dag_to_spec, node_succ,
                            brute_paths_between)
import workloads as W


def _groups(spec, **kw):
    gs, _ = P.groups(spec, P.Options(**kw))
    return sorted(gs.values())


def test_worked_example_one_group():
    g, expect = graph_from_golden("fuseops_worked_example.txt")
    gs = _groups(g)
    node = g.node_of_value()
    assert gs == [[node[v] for v in expect["expect_groups"]]]
    leaves, out, _ = P.group_io(g, gs[0])
    assert leaves == expect["expect_leaves"] and out == 4


def test_diamond_one_group():
    assert _groups(W.diamond(64, 32)) == [list(range(7))]


def test_matmul_diamond_phase0():
    """The page's diamond drawn with conv2d as producer: a kOutEWiseFusable op
    fuses with its elementwise post-dominator across elementwise branches."""
    g = W.GraphSpec()
    a = g.input((8, 16), "bf16")
    b = g.input((16, 8), "bf16")
    m = g.op("matmul_bf16", (a, b), (0, 0))
    r1 = g.op("relu", (m,))
    r2 = g.op("exp", (m,))
    r3 = g.op("tanh", (m,))
    s = g.op("add", (r1, r2, r3))
    g.mark_output(s)
    assert _groups(g) == [[0, 1, 2, 3, 4]]


def test_matmul_bias_relu_one_group():
    """conv2d + bias_add + relu pattern (phase 0), matmul standing for conv2d."""
    g = W.GraphSpec()
    a = g.input((8, 16), "bf16")
    b = g.input((16, 8), "bf16")
    bias = g.input((8,))
    m = g.op("matmul_bf16", (a, b), (0, 0))
    ba = g.op("badd_col", (m, bias))
    r = g.op("relu", (ba,))
    g.mark_output(r)
    assert _groups(g) == [[0, 1, 2]]


def test_two_matmuls_never_fuse():
    g = W.GraphSpec()
    a = g.input((8, 8), "bf16")
    b = g.input((8, 8), "bf16")
    m1 = g.op("matmul_bf16", (a, b), (0, 0))
    m2 = g.op("matmul_bf16", (m1, b), (0, 0))
    g.mark_output(m2)
    assert _groups(g) == [[0], [1]]


def test_sf_update_one_group():
    assert _groups(W.sf_update(64, 32, 32)) == [list(range(6))]


def test_reduce_is_a_sink_only():
    g = W.rnnlm_chain(8, 16)
    assert _groups(g) == [[0, 1, 2], [3]]
    # DisCo-style predecessor fusion: the reduce group takes the sigmoid
    assert _groups(g, allow_reduce_epilogue=True) == [[0, 1, 2, 3]]


def test_opaque_is_a_barrier():
    g = W.GraphSpec()
    x = g.input((4, 4))
    a = g.op("relu", (x,))
    b = g.op("opaque_copy", (a,))
    c = g.op("exp", (b,))
    d = g.op("tanh", (c,))
    g.mark_output(d)
    assert _groups(g) == [[0], [1], [2, 3]]


def test_max_fused_ops_256():
    g = W.GraphSpec()
    v = g.input((4, 4))
    for _ in range(300):
        v = g.op("relu", (v,))
    g.mark_output(v)
    gs = _groups(g)
    assert [len(x) for x in gs] == [256, 44]
    assert [len(x) for x in _groups(g, max_fused_ops=100)] == [100, 100, 100]


def test_max_args():
    """Each add reads a fresh input; with max_args=4 a group holds at most 3
    distinct outside values."""
    g = W.GraphSpec()
    v = g.input((4, 4))
    for _ in range(6):
        v = g.op("add", (v, g.input((4, 4))))
    g.mark_output(v)
    gs = _groups(g, max_args=4)
    for grp in gs:
        leaves, _, _ = P.group_io(g, grp)
        assert len(leaves) + 1 <= 4
    assert len(gs) > 1
    assert len(_groups(g)) == 1


def test_injective_waits_for_phase_1():
    """transpose -> relu: relu's group is elementwise, the transpose injective;
    the transpose joins its elementwise post-dominator only in phase 1."""
    g = W.GraphSpec()
    x = g.input((4, 8))
    t = g.op("transpose", (x,))
    r = g.op("relu", (t,))
    g.mark_output(r)
    assert _groups(g) == [[0, 1]]


def test_injective_does_not_enter_reduce():
    g = W.GraphSpec()
    x = g.input((4, 8))
    t = g.op("transpose", (x,))
    s = g.op("rowsum", (t,))
    g.mark_output(s)
    assert _groups(g) == [[0], [1]]


def _check_invariants(spec, gs, allow_epi=False):
    node_vid, succ, exits = node_succ(spec)
    n = len(node_vid)
    group_of = {}
    for sink, nodes in gs.items():
        for i in nodes:
            group_of[i] = sink
    for sink, nodes in gs.items():
        S = set(nodes)
        assert max(nodes) == sink
        # exactly one node whose value leaves the group: the sink
        escaping = [i for i in nodes if exits[i] or any(group_of[c] != sink for c in succ[i])]
        assert escaping == [sink], (nodes, escaping)
        # convex: every path between two members stays inside
        for a in nodes:
            for b in nodes:
                if a < b:
                    for path in brute_paths_between(succ, a, b):
                        assert set(path) <= S
        # at most one anchor; a reduce is the sink unless an epilogue is allowed
        kk = [kinds.op_kind(spec.values[node_vid[i]].op) for i in nodes]
        assert sum(k in (kinds.K_COMM_REDUCE, kinds.K_OUT_EWISE_FUSABLE) for k in kk) <= 1
        if not allow_epi:
            for i, k in zip(nodes, kk):
                if k == kinds.K_COMM_REDUCE:
                    assert i == sink
        if kinds.K_OPAQUE in kk:
            assert len(nodes) == 1
    assert sorted(group_of) == list(range(n))


def test_invariants_random_small_dags():
    rng = np.random.default_rng(3)
    for n, preds in small_dags(7, seed=5, count=1500):
        ops = rng.integers(0, 5, size=n)
        spec = dag_to_spec(n, preds, ops)
        gs, _ = P.groups(spec)
        _check_invariants(spec, gs)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_invariants_random_dag_workload(seed):
    spec = W.random_dag(seed, **W.CONFIGS["random_dag"]["small"])
    gs, _ = P.groups(spec)
    _check_invariants(spec, gs)
    # same topology at full size -> same partition
    full = W.random_dag(seed)
    assert P.groups(full)[0] == gs


# ---- tuples and phase 2 (TVM "Operator Fusion", Fusion rules) ---------------
def _inception():
    """Two branches joined by a tuple and a concatenation, then a tail."""
    g = W.GraphSpec()
    x1 = g.input((64, 32))
    x2 = g.input((32, 32))
    a = g.op("relu", (x1,))
    b = g.op("exp", (x2,))
    t = g.op("tuple", (a, b))
    c = g.op("concat", (t,))
    s = g.op("scale", (c,), (0.5,))
    g.mark_output(s)
    return g


def test_phase1_absorbs_the_tuple_phase2_its_fields():
    from oracle import partition as OP
    spec = _inception()
    group_of, ipdom = OP.partition(spec)
    # the tuple fuses into the concat and its tail (phase 1); the branches,
    # blocked by the tuple edge in phases 0 and 1, join in phase 2
    assert ipdom[:2] == [2, 2]
    assert group_of == [4, 4, 4, 4, 4]


def test_phase2_only_after_absorption():
    from oracle import partition as OP
    g = W.GraphSpec()
    x1 = g.input((16, 8))
    x2 = g.input((16, 8))
    a = g.op("relu", (x1,))
    b = g.op("neg", (x2,))
    t = g.op("tuple", (a, b))
    r = g.op("rowsum", (t,))          # a tuple does not fuse into a reduction
    g.mark_output(r)
    group_of, _ = OP.partition(g)
    assert group_of == [0, 1, 2, 3]


def test_phase2_path_must_be_injective_or_simpler():
    from oracle import partition as OP
    g = W.GraphSpec()
    x1 = g.input((16, 8))
    x2 = g.input((8, 16))
    a = g.op("exp", (x1,))
    tr = g.op("transpose", (x2,))    # injective: joins through phase 2
    t = g.op("tuple", (a, tr))
    c = g.op("concat", (t,))
    o = g.op("relu", (c,))
    g.mark_output(o)
    group_of, _ = OP.partition(g)
    assert group_of == [4, 4, 4, 4, 4]


def test_phase2_skips_a_matmul_field():
    from oracle import partition as OP
    g = W.GraphSpec()
    x = g.input((16, 8), "bf16")
    w = g.input((8, 8), "bf16")
    y = g.input((16, 8))
    m = g.op("matmul_bf16", (x, w), (0, 0))   # out-elementwise-fusable: never phase 2
    r = g.op("relu", (y,))
    t = g.op("tuple", (m, r))
    c = g.op("concat", (t,))
    g.mark_output(c)
    group_of, _ = OP.partition(g)
    assert group_of == [0, 3, 3, 3]
