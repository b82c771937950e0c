"""Pins for the oracle's pattern-based grouping (TVM "Operator Fusion",
FuseOpsByPattern): the page's matmul + bias example, priority order, the
private-intermediate check, convexity, and the invariants of a match set on
random graphs."""
import numpy as np
import pytest

import workloads as W
from oracle import patterns as PT


def _mlp():
    g = W.GraphSpec()
    x = g.input((64, 32), "bf16")
    w = g.input((32, 48), "bf16")
    b = g.input((48,))
    m = g.op("matmul_bf16", (x, w), (0, 0))
    a = g.op("badd_col", (m, b))
    r = g.op("relu", (a,))
    s = g.op("scale", (r,), (2.0,))
    g.mark_output(s)
    return g


MB = ("cutlass.matmul_bias", ["matmul_bf16", "badd_col"], True)
MBR = ("cutlass.matmul_bias_relu", ["matmul_bf16", "badd_col", "relu"], True)


def test_page_example_matmul_bias():
    groups, mo = PT.match(_mlp(), [MB])
    assert groups == [[0, 1], [2], [3]] and mo == [0, 0, -1, -1]


def test_first_pattern_wins():
    assert PT.match(_mlp(), [MBR, MB])[0] == [[0, 1, 2], [3]]
    assert PT.match(_mlp(), [MB, MBR])[0] == [[0, 1], [2], [3]]


def test_private_check_rejects_shared_intermediates():
    g = _mlp()
    g.mark_output(g.ops[0].vid)            # the matmul's result is also returned
    assert PT.match(g, [MB])[0] == [[0], [1], [2], [3]]
    assert PT.match(g, [(MB[0], MB[1], False)])[0] == [[0, 1], [2], [3]]


def test_non_convex_chain_is_rejected():
    g = W.GraphSpec()
    x = g.input((8, 8))
    a = g.op("relu", (x,))
    y = g.op("exp", (a,))                  # leaves {relu, add} ...
    z = g.op("add", (a, y))                # ... and comes back
    g.mark_output(z)
    assert PT.match(g, [("p", ["relu", "add"], False)])[0] == [[0], [1], [2]]
    assert PT.match(g, [("p", ["relu", "exp", "add"], False)])[0] == [[0, 1, 2]]


def test_a_taken_operator_joins_no_second_match():
    g = W.GraphSpec()
    x = g.input((8, 8))
    a = g.op("relu", (x,))
    b = g.op("relu", (x,))
    c = g.op("add", (a, b))
    g.mark_output(c)
    groups, mo = PT.match(g, [("p", ["relu", "add"], False)])
    assert groups == [[0, 2], [1]] and mo == [0, -1, 0]


@pytest.mark.parametrize("seed", range(20))
def test_match_invariants_on_random_graphs(seed):
    from tests._helpers import small_dags, dag_to_spec
    r = np.random.default_rng(seed)
    n, preds = next(iter(small_dags(9, seed=900 + seed, count=1)))
    spec = dag_to_spec(n, preds, op_choice=[int(x) for x in r.integers(0, 2, size=n)], outputs=[n - 1])
    pats = [("a", ["relu", "add"], True), ("b", ["add", "mul"], False), ("c", ["transpose", "relu"], True),
            ("d", ["relu", "relu"], False)]
    groups, mo = PT.match(spec, pats)
    assert sorted(x for g in groups for x in g) == list(range(n))
    node_of = spec.node_of_value()
    for g in groups:
        if len(g) == 1 and mo[g[0]] < 0:
            continue
        k = mo[g[0]]
        assert all(mo[x] == k for x in g)
        chain = pats[k][1]
        assert sorted(spec.ops[x].op for x in g) == sorted(chain)
        # each member after the first reads another member's output
        for x in g:
            if spec.ops[x].op != chain[0] or x != g[0]:
                assert any(node_of.get(a) in g for a in spec.ops[x].args)
