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
