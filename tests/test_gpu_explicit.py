"""GPU parity of plans built from explicit fusion moves (DisCo, Introduction:
non-duplicate fusion gives a group extra outputs, duplicate fusion a copy of
the predecessor): every value a group writes, against the oracle, through the
C ABI."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import explicit as OX
from oracle import execute as OE
from tests._helpers import rel_err, check_parity, TOL_F32, small_dags, dag_to_spec
from tests._gpu import to_dev, run_fused
from group_execution_gb300 import graph_from_spec, _lib, FgError

pytestmark = pytest.mark.gpu


def _run_moves(spec, moves, from_fuseops=False, seed=0, expect_outs=None):
    g = graph_from_spec(spec)
    part = g.partition(from_fuseops=from_fuseops)
    st = OX.initial(spec, from_fuseops=from_fuseops)
    for node, pred, dup in moves:
        part.fuse(node, pred, dup)
        st = OX.fuse(st, node, pred, dup)
    assert part.query() == (st.label, st.clone_of)
    plan = part.build()
    order = OX.groups(st)
    assert [sorted(gi.nodes) for gi in plan.groups] == [sorted(x) for x in order]
    ins = W.make_inputs(spec, seed)
    dev = {vid: to_dev(spec, vid, a) for vid, a in ins.items()}
    env = run_fused(plan, spec, dev)
    plan.sync()
    ref = OE.run_unfused(spec, ins, keep=[v.vid for v in spec.ops])
    written = [o for gi in plan.groups for o in gi.outs]
    for o in written:
        check_parity(spec, o, env[o].cpu().numpy(), ref[o])
    if expect_outs is not None:
        assert [gi.outs for gi in plan.groups] == expect_outs
    return plan


@pytest.mark.parametrize("shape", [(64, 32), (200, 132), (33, 96), (8192, 4096)])
def test_diamond_multi_output_and_copy(shape):
    spec = W.diamond(*shape)
    # P = X + bias into relu's group (P stays an output: the scale and the
    # multiply read it), a copy of P into the scale's group, then exp into
    # the scale's group and the 3-way add with the multiply
    plan = _run_moves(spec, [(1, 0, False), (2, 0, True), (3, 2, False), (5, 4, False)])
    assert any(len(gi.outs) > 1 for gi in plan.groups)


def test_transposed_extra_output():
    g = W.GraphSpec()
    x = g.input((96, 160))
    a = g.op("relu", (x,))
    t = g.op("transpose", (a,))
    b = g.op("exp", (g.op("scale", (t,), (0.01,)),))
    c = g.op("scale", (a,), (2.0,))
    g.mark_output(b)
    g.mark_output(c)
    # {relu, transpose, scale, exp}: the frame is [160, 96]; relu's output,
    # read by the other scale, is written through the transposed map
    plan = _run_moves(g, [(1, 0, False), (2, 1, False), (3, 2, False)])
    assert plan.groups[0].outs == [b, a]


def test_permuted_extra_output():
    g = W.GraphSpec()
    x = g.input((64, 96))
    a = g.op("relu", (x,))
    t = g.op("transpose", (a,))
    r = g.op("reshape", (t,), (48, 128))
    b = g.op("exp", (g.op("scale", (r,), (0.01,)),))
    c = g.op("neg", (a,))
    g.mark_output(b)
    g.mark_output(c)
    # frame [48, 128]; relu's output is a digit permutation of it (neither
    # the identity nor the transpose)
    plan = _run_moves(g, [(1, 0, False), (2, 1, False), (3, 2, False), (4, 3, False)])
    assert plan.groups[0].outs == [b, a]


def test_reduce_group_with_prologue_output():
    g = W.GraphSpec()
    x = g.input((300, 1024))
    y = g.input((300, 1024))
    w = g.input((1024,))
    a = g.op("mul", (x, y))
    b = g.op("bmul_col", (a, w))
    s = g.op("rowsum", (b,))
    o = g.op("sigmoid", (s,))
    c = g.op("relu", (a,))
    g.mark_output(o)
    g.mark_output(c)
    plan = _run_moves(g, [(1, 0, False), (2, 1, False)])
    red = [gi for gi in plan.groups if gi.kind == "reduce"][0]
    assert red.outs == [s, a]


@pytest.mark.parametrize("seed", range(8))
def test_random_moves(seed):
    r = np.random.default_rng(seed)
    n, preds = next(iter(small_dags(8, seed=500 + seed, count=1)))
    spec = dag_to_spec(n, preds, op_choice=[int(x) for x in r.integers(0, 2, size=n)], outputs=[n - 1])
    part = graph_from_spec(spec).partition(from_fuseops=bool(seed % 2))
    st = OX.initial(spec, from_fuseops=bool(seed % 2))
    moves = []
    for _ in range(12):
        node = int(r.integers(0, len(st.ops)))
        prod = {o[3]: i for i, o in enumerate(st.ops)}
        cands = [prod[a] for a in st.ops[node][1] if a in prod]
        if not cands:
            continue
        mv = (node, cands[int(r.integers(0, len(cands)))], bool(r.integers(0, 2)))
        try:
            nxt = OX.fuse(st, *mv)
            part.fuse(*mv)
        except (ValueError, OX.NotConvex, FgError):
            continue
        st = nxt
        moves.append(mv)
    _run_moves(spec, moves, from_fuseops=bool(seed % 2), seed=seed)


def _mlp_spec(M, K, N):
    g = W.GraphSpec()
    x = g.input((M, K), "bf16")
    w = g.input((K, N), "bf16")
    b = g.input((N,))
    m = g.op("matmul_bf16", (x, w), (0, 0))
    a = g.op("badd_col", (m, b))
    r = g.op("relu", (a,))
    s = g.op("scale", (r,), (0.5,))
    g.mark_output(s)
    return g


def test_pattern_mlp_full_size():
    """The MLP layer the benchmark times, relu(X W + b) with X, W [4096, 4096]
    bf16: the matmul + bias + relu pattern makes it one GEMM-epilogue group,
    launched as the benchmark launches it, the whole output against the
    oracle."""
    spec = W.GraphSpec()
    x = spec.input((4096, 4096), "bf16")
    w = spec.input((4096, 4096), "bf16")
    b = spec.input((4096,))
    y = spec.op("relu", (spec.op("badd_col", (spec.op("matmul_bf16", (x, w), (0, 0)), b)),))
    spec.mark_output(y)
    plan = graph_from_spec(spec).partition(patterns=[("matmul_bias_relu", ["matmul_bf16", "badd_col", "relu"], True)]).build()
    assert plan.n_groups == 1 and plan.groups[0].kind == "gemm"
    ins = W.make_inputs(spec, 0)
    dev = {vid: to_dev(spec, vid, a) for vid, a in ins.items()}
    env = run_fused(plan, spec, dev)
    plan.sync()
    ref = OE.run_unfused(spec, ins)[y]
    assert rel_err(env[y].cpu().numpy(), ref) <= 1e-4


@pytest.mark.parametrize("shape", [(256, 128, 512), (200, 72, 264)])
def test_pattern_plan_matmul_bias_relu(shape):
    """FuseOpsByPattern with the page's matmul + bias pattern extended by relu:
    the match runs as one GEMM-epilogue group, the scale alone."""
    from oracle import patterns as PT
    spec = _mlp_spec(*shape)
    pats = [("matmul_bias_relu", ["matmul_bf16", "badd_col", "relu"], True)]
    part = graph_from_spec(spec).partition(patterns=pats)
    assert part.match_of == PT.match(spec, pats)[1] == [0, 0, 0, -1]
    plan = part.build()
    assert [sorted(gi.nodes) for gi in plan.groups] == [[0, 1, 2], [3]]
    ins = W.make_inputs(spec, 0)
    dev = {vid: to_dev(spec, vid, a) for vid, a in ins.items()}
    env = run_fused(plan, spec, dev)
    plan.sync()
    ref = OE.run_unfused(spec, ins, keep=[v.vid for v in spec.ops])
    for gi in plan.groups:
        for o in gi.outs:
            assert rel_err(env[o].cpu().numpy(), ref[o]) <= 1e-4
