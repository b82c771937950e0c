"""Host-side checks of the C ABI (no GPU needed): the library loads and exports
every declared symbol, graph construction validates its input, and the C++
grouping (post-dominator tree and FuseOps phases) equals the oracle's
bit for bit, down to each group's leaves and algorithmic bytes."""
import ctypes as C

import pytest

import workloads as W
from oracle import partition as OP
from group_execution_gb300 import _lib, graph_from_spec, Graph, FgError
from tests._helpers import graph_from_golden


def test_library_exports_every_header_symbol():
    lib = _lib.load()
    names = _lib.header_symbols()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES)


def _parity(spec, **kw):
    g = graph_from_spec(spec)
    plan = g.build(**kw)
    ref_group_of, ref_ipdom = OP.partition(spec, OP.Options(
        max_fused_ops=kw.get("max_fused_ops", 256), max_args=kw.get("max_args", 64),
        allow_reduce_epilogue=kw.get("allow_reduce_epilogue", False)))
    assert plan.ipdom == ref_ipdom
    assert plan.group_of == ref_group_of
    ref_groups, _ = OP.groups(spec, OP.Options(
        max_fused_ops=kw.get("max_fused_ops", 256), max_args=kw.get("max_args", 64),
        allow_reduce_epilogue=kw.get("allow_reduce_epilogue", False)))
    sinks = sorted(ref_groups)
    assert plan.n_groups == len(sinks)
    for gid, s in enumerate(sinks):
        info = plan.groups[gid]
        leaves, out, alg = OP.group_io(spec, ref_groups[s])
        assert info.nodes == ref_groups[s]
        assert info.leaves == leaves and info.out == out and info.alg_bytes == alg
    return plan


@pytest.mark.parametrize("name", ["rnnlm_chain", "diamond", "sf_update"])
def test_config_partitions(name):
    for size in ("small", "full"):
        spec = getattr(W, name)(**W.CONFIGS[name][size])
        _parity(spec)
        _parity(spec, allow_reduce_epilogue=True)


def test_partition_groups_of_the_configs():
    assert graph_from_spec(W.diamond(64, 32)).build().n_groups == 1
    assert graph_from_spec(W.sf_update(64, 32, 32)).build().n_groups == 1
    assert graph_from_spec(W.rnnlm_chain()).build().n_groups == 2
    assert graph_from_spec(W.rnnlm_chain()).build(allow_reduce_epilogue=True).n_groups == 1


def test_worked_example_through_the_abi():
    spec, expect = graph_from_golden("fuseops_worked_example.txt")
    plan = _parity(spec)
    assert plan.n_groups == 1 and plan.groups[0].leaves == expect["expect_leaves"]


@pytest.mark.parametrize("seed", range(12))
def test_random_dag_partition_bit_exact(seed):
    spec = W.random_dag(seed, **W.CONFIGS["random_dag"]["small"])
    _parity(spec)
    _parity(spec, allow_reduce_epilogue=True)
    _parity(spec, max_fused_ops=5, max_args=4)


@pytest.mark.parametrize("n_ops", [10, 30, 60])
def test_random_dag_sizes(n_ops):
    for seed in range(20):
        spec = W.random_dag(100 + seed, n_ops=n_ops, R=16, C=8, nominal_R=8192, nominal_C=4096)
        _parity(spec)
        _parity(spec, max_fused_ops=3)


def test_full_size_random_dags():
    for seed in range(4):
        _parity(W.random_dag(seed))


def test_long_chain_size_limit():
    g = W.GraphSpec()
    v = g.input((4, 4))
    for _ in range(300):
        v = g.op("relu", (v,))
    g.mark_output(v)
    plan = _parity(g)
    assert [len(x.nodes) for x in plan.groups] == [256, 44]


def test_graph_validation_errors():
    g = Graph()
    x = g.input((4, 8))
    v = g.input((8,))
    u = g.input((8, 4), "bf16")
    with pytest.raises(FgError) as e:
        g.op("add", (x, v))
    assert e.value.status == _lib.FG_ESHAPE
    with pytest.raises(FgError) as e:
        g.op("badd_row", (x, v))
    assert e.value.status == _lib.FG_ESHAPE
    with pytest.raises(FgError) as e:
        g.op("relu", (u,))
    assert e.value.status == _lib.FG_EUNSUPPORTED
    with pytest.raises(FgError) as e:
        g.op("reshape", (x,), (3, 11))
    assert e.value.status == _lib.FG_ESHAPE
    with pytest.raises(FgError) as e:
        g.op("matmul_bf16", (x, x), (0, 0))
    assert e.value.status == _lib.FG_EINVAL
    with pytest.raises(FgError) as e:
        g.op("relu", (99,))
    assert e.value.status == _lib.FG_EINVAL
    lib = _lib.load()
    vid = C.c_int32()
    assert lib.fg_graph_add_op(g.h, 999, 1, (C.c_int32 * 1)(x), 0, None, C.byref(vid)) == _lib.FG_EINVAL
    assert b"opcode" in lib.fg_last_error()
    assert lib.fg_graph_add_op(None, 0, 0, None, 0, None, C.byref(vid)) == _lib.FG_EINVAL
    assert lib.fg_build_groups(None, None, None) == _lib.FG_EINVAL


def test_plan_query_errors():
    spec = W.diamond(16, 8)
    plan = graph_from_spec(spec).build()
    lib = _lib.load()
    assert lib.fg_plan_group_info(plan.h, 5, None, None, None, None, None, None, None, None) == _lib.FG_EINVAL
    assert lib.fg_launch_group(plan.h, -1, None, None) == _lib.FG_EINVAL
    assert lib.fg_launch_unfused(plan.h, 99, None, None) == _lib.FG_EINVAL


def test_exec_info_of_the_diamond():
    plan = graph_from_spec(W.diamond(8192, 4096)).build()
    info = plan.exec_info(0)
    assert info["n_staged"] == 3 and info["n_gathered"] == 0
    assert info["stages"] >= 3
    assert plan.groups[0].alg_bytes == 2 * 8192 * 4096 * 4 + 4096 * 4 + 8192 * 4096 * 4


# ---- AllReduce bucket planning (host side of the C ABI) ----------------------
def test_plan_threshold_matches_oracle():
    import numpy as np
    from oracle import buckets as OB
    from group_execution_gb300 import plan_threshold
    r = np.random.default_rng(11)
    cases = [(W.tensor_fusion_sizes(0), T) for T in (0, 1 << 20, 4 << 20, 16 << 20, 1 << 40)]
    for _ in range(200):
        n = int(r.integers(0, 40))
        cases.append((r.integers(0, 50_000, size=n), int(r.integers(0, 300_000))))
    for sizes, T in cases:
        for dt, eb in (("bf16", 2), ("f32", 4)):
            for align in (16, 256, 4096):
                got = plan_threshold(list(sizes), T, dt, align)
                assert got == OB.threshold_buckets(list(sizes), T, eb, align), (len(sizes), T, dt, align)


def test_buckets_merge_matches_oracle():
    from oracle import buckets as OB
    from group_execution_gb300 import merge_buckets
    b = [0, 2, 7, 8, 20]
    for j in range(len(b) - 2):
        assert merge_buckets(b, j) == OB.merge_neighbours(b, j)
    with pytest.raises(FgError):
        merge_buckets(b, len(b) - 2)


def test_plan_threshold_rejects_bad_arguments():
    from group_execution_gb300 import plan_threshold
    with pytest.raises(FgError):
        plan_threshold([1, 2], 100, align=24)
    with pytest.raises(FgError):
        plan_threshold([1, -2], 100)
    with pytest.raises(FgError):
        plan_threshold([1, 2], -1)


# ---- explicit fusion moves (host side of the C ABI) --------------------------
def _lib_moves_match_oracle(spec, seed, from_fuseops):
    import numpy as np
    from oracle import explicit as OX
    from group_execution_gb300 import _lib as L
    r = np.random.default_rng(seed)
    part = graph_from_spec(spec).partition(from_fuseops=from_fuseops)
    st = OX.initial(spec, from_fuseops=from_fuseops)
    assert part.query() == (st.label, st.clone_of)
    accepted = 0
    for _ in range(16):
        node = int(r.integers(0, len(st.ops)))
        prod = {o[3]: i for i, o in enumerate(st.ops)}
        cands = [prod[a] for a in st.ops[node][1] if a in prod]
        pred = cands[int(r.integers(0, len(cands)))] if cands and r.random() < 0.9 else int(r.integers(0, len(st.ops)))
        dup = bool(r.integers(0, 2))
        try:
            nxt, why = OX.fuse(st, node, pred, dup), None
        except ValueError:
            nxt, why = None, L.FG_EINVAL
        except OX.NotConvex:
            nxt, why = None, L.FG_EUNSUPPORTED
        try:
            part.fuse(node, pred, dup)
            ok = True
        except FgError as e:
            ok, status, msg = False, e.status, str(e)
        if nxt is None:
            assert not ok and status == why, (node, pred, dup)
            continue
        if not ok:
            # the library may refuse a convex move its kernels cannot run
            assert status == L.FG_EUNSUPPORTED and "convex" not in msg, msg
            continue
        st = nxt
        accepted += 1
        assert part.query() == (st.label, st.clone_of), (node, pred, dup)
    return accepted


def test_partition_moves_match_oracle():
    from tests._helpers import small_dags, dag_to_spec
    import numpy as np
    total = 0
    for k, (n, preds) in enumerate(small_dags(8, seed=77, count=120)):
        r = np.random.default_rng(k)
        # relu / transpose, add / mul: every operator of the random DAGs is legal in the library
        spec = dag_to_spec(n, preds, op_choice=[int(x) for x in r.integers(0, 2, size=n)], outputs=[n - 1])
        total += _lib_moves_match_oracle(spec, k, from_fuseops=bool(k % 2))
    assert total > 100


def test_partition_moves_on_the_workloads():
    for spec in (W.rnnlm_chain(), W.diamond(64, 32), W.sf_update(64, 128, 256)):
        _lib_moves_match_oracle(spec, 1, False)
        _lib_moves_match_oracle(spec, 2, True)


def test_partition_plan_groups_follow_dependencies():
    from oracle import explicit as OX
    spec = W.diamond(64, 32)
    g = graph_from_spec(spec)
    part = g.partition(from_fuseops=False)
    st = OX.initial(spec, from_fuseops=False)
    # relu, the scale and the multiply all read P = X + bias: fold P into
    # relu's group without copying (P becomes an extra output), copy it into
    # the scale's group
    for node, pred, dup in ((1, 0, False), (2, 0, True)):
        part.fuse(node, pred, dup)
        st = OX.fuse(st, node, pred, dup)
    assert part.query() == (st.label, st.clone_of)
    plan = part.build()
    order = OX.groups(st)
    assert [sorted(gi.nodes) for gi in plan.groups] == [sorted(x) for x in order]
    for gi, nodes in zip(plan.groups, order):
        assert gi.outs == OX.group_outputs(st, nodes)


def test_interpreter_refuses_extra_outputs():
    from group_execution_gb300 import _lib as L
    spec = W.diamond(64, 32)
    part = graph_from_spec(spec).partition(from_fuseops=False, flags=L.FG_FLAG_INTERPRET)
    with pytest.raises(FgError) as e:
        part.fuse(1, 0, False)     # P keeps other readers: an extra output
    assert e.value.status == L.FG_EUNSUPPORTED
    part.fuse(2, 0, True)          # a copy needs no extra output


def test_opaque_operators_stay_alone():
    g = W.GraphSpec()
    x = g.input((8, 8))
    a = g.op("opaque_copy", (x,))
    b = g.op("relu", (a,))
    g.mark_output(b)
    part = graph_from_spec(g).partition(from_fuseops=False)
    with pytest.raises(FgError):
        part.fuse(1, 0, False)


# ---- training-step simulator (host side of the C ABI) ------------------------
def test_simulate_matches_oracle():
    import numpy as np
    from oracle import simulate as OS
    from group_execution_gb300 import simulate
    for seed in range(300):
        r = np.random.default_rng(seed)
        n = int(r.integers(1, 40))
        edges = sorted({(int(a), int(b)) for a, b in r.integers(0, n, size=(2 * n, 2)) if a < b})
        times = r.uniform(0.1, 3.0, size=n).tolist()
        nt = int(r.integers(0, 20))
        prod = r.integers(0, n, size=nt).tolist()
        by = r.uniform(1, 1e6, size=nt).tolist()
        order = r.permutation(nt).tolist()
        cuts = sorted(set(r.integers(0, nt + 1, size=4).tolist()) | {0, nt})
        buckets = [order[a:b] for a, b in zip(cuts, cuts[1:]) if b > a]
        ar_edges = [(int(b), int(t)) for b, t in zip(r.integers(0, max(1, len(buckets)), size=3),
                                                       r.integers(0, n, size=3))
                    if len(buckets) and all(prod[x] < t for x in buckets[int(b)])]
        c, d = float(r.uniform(1e-7, 1e-5)), float(r.uniform(0, 1))
        got = simulate(times, edges, prod, by, buckets, c, d, ar_edges)
        ref = OS.simulate(times, edges, prod, by, buckets, c, d, ar_edges)
        assert got[0] == ref[0] and got[1] == ref[1] and got[2] == ref[2] and got[3] == ref[3], seed


def test_simulate_rejects_cycles_and_bad_ids():
    from group_execution_gb300 import simulate
    with pytest.raises(FgError):
        simulate([1, 1], [(0, 1), (1, 0)], [], [], [], 0.0, 0.0)
    with pytest.raises(FgError):
        simulate([1], [(0, 3)], [], [], [], 0.0, 0.0)
    with pytest.raises(FgError):
        simulate([1], [], [2], [1.0], [[0]], 0.0, 0.0)


# ---- pattern-based grouping (host side of the C ABI) -------------------------
def _labels(groups, n):
    lab = [0] * n
    for g in groups:
        for x in g:
            lab[x] = min(g)
    return lab


def test_patterns_match_oracle():
    import numpy as np
    from oracle import patterns as PT
    from tests._helpers import small_dags, dag_to_spec
    pats = [("a", ["relu", "add"], True), ("b", ["add", "mul"], False), ("c", ["transpose", "relu"], True),
            ("d", ["relu", "relu"], False), ("e", ["mul", "relu", "add"], False)]
    for k, (n, preds) in enumerate(small_dags(9, seed=31, count=200)):
        r = np.random.default_rng(k)
        spec = dag_to_spec(n, preds, op_choice=[int(x) for x in r.integers(0, 2, size=n)], outputs=[n - 1])
        order = r.permutation(len(pats)).tolist()
        use = [pats[i] for i in order[:int(r.integers(1, len(pats) + 1))]]
        groups, mo = PT.match(spec, use)
        part = graph_from_spec(spec).partition(patterns=use)
        assert part.match_of == mo, k
        assert part.query()[0] == _labels(groups, n), k


def test_page_pattern_matmul_bias():
    from oracle import patterns as PT
    g = W.GraphSpec()
    x = g.input((256, 128), "bf16")
    w = g.input((128, 512), "bf16")
    b = g.input((512,))
    m = g.op("matmul_bf16", (x, w), (0, 0))
    a = g.op("badd_col", (m, b))
    rl = g.op("relu", (a,))
    g.mark_output(rl)
    pats = [("cutlass.matmul_bias", ["matmul_bf16", "badd_col"], True)]
    part = graph_from_spec(g).partition(patterns=pats)
    assert part.match_of == PT.match(g, pats)[1] == [0, 0, -1]
    plan = part.build()
    assert [sorted(gi.nodes) for gi in plan.groups] == [[0, 1], [2]]
    assert plan.groups[0].kind == "gemm"


@pytest.mark.parametrize("seed", range(60))
def test_partition_with_tuples_matches_oracle(seed):
    from tests._helpers import tuple_dag
    _parity(tuple_dag(seed))


def test_launches_fail_loudly_without_a_device():
    """With no CUDA device every entry point that would run a kernel returns
    FG_ECUDA (there is no CPU fallback), while graph building and grouping
    still work; the tensor-fusion calls refuse a null layout with FG_EINVAL.
    Pointers here are never dereferenced: each call fails before any launch."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    lib = _lib.load()
    spec = W.diamond(200, 132)
    plan = graph_from_spec(spec).build()
    info = plan.groups[0]
    ptrs = plan._ptrs({v: 0x100000 * (i + 1) for i, v in enumerate(info.leaves + info.outs)})
    assert lib.fg_launch_group(plan.h, 0, ptrs, None) == _lib.FG_ECUDA
    assert lib.fg_launch_unfused(plan.h, 0, ptrs, None) == _lib.FG_ECUDA
    assert lib.fg_sync_status(plan.h, None) == _lib.FG_ECUDA
    numel = (C.c_int64 * 2)(10, 20)
    grads = (C.c_void_p * 2)(0x100000, 0x200000)
    h, offs, total = C.c_void_p(), (C.c_int64 * 2)(), C.c_int64()
    assert lib.tf_layout_create(2, numel, grads, _lib.FG_BF16, 256, C.byref(h), offs, C.byref(total)) == _lib.FG_ECUDA
    assert h.value is None
    rowsum = _lib.OPCODES["rowsum"]
    assert lib.fg_row_reduce_noalloc(rowsum, C.c_void_p(0x100000), 4, 8, C.c_void_p(0x200000), None) == _lib.FG_ECUDA
    assert lib.fg_row_reduce_noalloc_status(None) == _lib.FG_ECUDA
    buf, ready = C.c_void_p(0x100000), C.c_int32()
    assert lib.tf_pack(None, C.c_float(1.0), buf, None) == _lib.FG_EINVAL
    assert lib.tf_unpack(None, C.c_float(1.0), buf, None) == _lib.FG_EINVAL
    assert lib.tf_layout_set_buckets(None, 1, (C.c_int32 * 2)(0, 2)) == _lib.FG_EINVAL
    assert lib.tf_pack_buckets(None, C.c_float(1.0), buf, None) == _lib.FG_EINVAL
    assert lib.tf_bucket_wait(None, 0, None) == _lib.FG_EINVAL
    assert lib.tf_bucket_ready(None, 0, C.byref(ready)) == _lib.FG_EINVAL
