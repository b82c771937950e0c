"""Pins for the oracle's explicit fusion moves (DisCo, Introduction: fusing
an operator with a predecessor, non-duplicate or duplicate).  Convexity is
checked against a transitive closure computed by matrix powers; the moves
against their definitions on small DAGs; execution of every transformed graph
against plain op-by-op execution of the original."""
import numpy as np
import pytest

import workloads as W
from oracle import explicit as OX
from oracle import execute as OE
from tests._helpers import small_dags, dag_to_spec


def _closure_convex(st, nodes):
    """Non-convex iff some outside node x has u ->* x ->* w with u, w inside
    (reachability by boolean matrix powers)."""
    n = len(st.ops)
    prod = {o[3]: i for i, o in enumerate(st.ops)}
    A = np.zeros((n, n), dtype=bool)
    for i, o in enumerate(st.ops):
        for a in o[1]:
            if a in prod:
                A[prod[a], i] = True
    R = A.copy()
    for _ in range(n):
        R = R | (R.astype(int) @ A.astype(int) > 0)
    inside = set(nodes)
    for x in range(n):
        if x in inside:
            continue
        if any(R[u, x] for u in inside) and any(R[x, w] for w in inside):
            return False
    return True


def test_convexity_matches_closure():
    r = np.random.default_rng(3)
    for n, preds in small_dags(7, seed=4, count=400):
        st = OX.initial(dag_to_spec(n, preds), from_fuseops=False)
        for _ in range(4):
            k = int(r.integers(1, n + 1))
            nodes = sorted(r.choice(n, size=k, replace=False).tolist())
            assert OX.is_convex(st, nodes) == _closure_convex(st, nodes), (preds, nodes)


def _random_moves(spec, st, r, count):
    applied = 0
    for _ in range(count):
        node = int(r.integers(0, len(st.ops)))
        prod = {o[3]: i for i, o in enumerate(st.ops)}
        preds = [prod[a] for a in st.ops[node][1] if a in prod]
        if not preds:
            continue
        pred = preds[int(r.integers(0, len(preds)))]
        dup = bool(r.integers(0, 2))
        try:
            st = OX.fuse(st, node, pred, dup)
            applied += 1
        except (ValueError, OX.NotConvex):
            continue
    return st, applied


@pytest.mark.parametrize("seed", range(30))
def test_moves_keep_groups_convex_ordered_and_values_unchanged(seed):
    r = np.random.default_rng(seed)
    n, preds = next(iter(small_dags(8, seed=100 + seed, count=1)))
    spec = dag_to_spec(n, preds, op_choice=[int(x) for x in r.integers(0, 2, size=n)],
                       outputs=[n - 1])
    st0 = OX.initial(spec, from_fuseops=bool(seed % 2))
    st, applied = _random_moves(spec, st0, r, 12)
    order = OX.groups(st)
    assert sorted(i for g in order for i in g) == list(range(len(st.ops)))
    prod = {o[3]: i for i, o in enumerate(st.ops)}
    placed = set()
    for g in order:
        assert _closure_convex(st, g)
        for i in g:                                   # every outside operand is ready
            for a in st.ops[i][1]:
                if a in prod and prod[a] not in g:
                    assert prod[a] in placed
        placed |= set(g)
    for i, c in enumerate(st.clone_of):               # copies repeat their original
        if c >= 0:
            assert st.ops[i][0] == st.ops[c][0] and st.ops[i][2] == st.ops[c][2]
            assert st.ops[i][1] == st0.ops[c][1]
    ins = W.make_inputs(spec, seed)
    env = OX.run(st, ins)
    ref = OE.run_unfused(spec, ins, keep=[v.vid for v in spec.ops])
    for vid, x in ref.items():
        np.testing.assert_array_equal(env[vid], x)


def _fork():
    """a = relu(x); b = exp(a); c = a + b: a has two readers."""
    g = W.GraphSpec()
    x = g.input((4, 4))
    a = g.op("relu", (x,))
    b = g.op("exp", (a,))
    c = g.op("add", (a, b))
    g.mark_output(c)
    return g


def test_non_duplicate_fusion_adds_the_predecessor_as_an_output():
    spec = _fork()
    st = OX.initial(spec, from_fuseops=False)
    st = OX.fuse(st, 1, 0, duplicate=False)           # exp with relu
    g = OX.members(st, st.label[0])
    assert g == [0, 1]
    # relu's value still feeds the add: it leaves the group as an extra output
    assert OX.group_outputs(st, g) == [spec.ops[1].vid, spec.ops[0].vid]
    assert [sorted(x) for x in OX.groups(st)] == [[0, 1], [2]]


def test_duplicate_fusion_copies_the_predecessor():
    spec = _fork()
    st = OX.initial(spec, from_fuseops=False)
    st = OX.fuse(st, 1, 0, duplicate=True)
    assert len(st.ops) == 4 and st.clone_of == [-1, -1, -1, 0]
    assert st.label == [0, 1, 2, 1]                   # the copy joins exp's group
    assert st.ops[1][1] == (st.ops[3][3],)            # exp reads the copy
    assert st.ops[2][1] == (spec.ops[0].vid, spec.ops[1].vid)   # add still reads the original
    assert OX.group_outputs(st, [1, 3]) == [spec.ops[1].vid]    # the copy is never materialised


def test_a_single_reader_makes_both_moves_the_same():
    spec = W.rnnlm_chain()
    st = OX.initial(spec, from_fuseops=False)
    a = OX.fuse(st, 1, 0, duplicate=False)            # Mul2 with Mul1 (DisCo Fig. 2)
    b = OX.fuse(st, 1, 0, duplicate=True)
    assert a.label == b.label == [0, 0, 2, 3] and len(b.ops) == 4
    assert OX.group_outputs(a, [0, 1]) == [spec.ops[1].vid]


def test_refused_moves():
    spec = _fork()
    st = OX.initial(spec, from_fuseops=False)
    with pytest.raises(ValueError):
        OX.fuse(st, 1, 2)                             # add is not a predecessor of exp
    # {relu, add} without exp: relu -> exp -> add leaves and re-enters
    with pytest.raises(OX.NotConvex):
        OX.fuse(st, 2, 0, duplicate=False)
    st2 = OX.fuse(st, 2, 0, duplicate=True)           # a copy of relu is fine
    assert st2.label[-1] == st2.label[2]
    st3 = OX.fuse(OX.fuse(st, 1, 0), 2, 1)
    with pytest.raises(ValueError):
        OX.fuse(st3, 2, 0)                            # already one group
