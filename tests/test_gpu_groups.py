"""GPU parity of the fused-group kernels (elementwise and reduce groups)
against the CPU oracle, element by element, through the C ABI."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import execute as OE
from tests._helpers import rel_err, check_parity, exact_value, TOL_F32
from tests._gpu import prepare, run_fused, run_unfused
from group_execution_gb300 import _lib, graph_from_spec

pytestmark = pytest.mark.gpu


# compiled programs (the small-group kernel for small groups), the
# interpreter, and compiled programs in the pipelined kernels only
MODES = [0, _lib.FG_FLAG_INTERPRET, _lib.FG_FLAG_NO_SMALL]


def _check(spec, seed=0, unfused=True, **kw):
    if "flags" not in kw:
        for fl in MODES:
            r = _check(spec, seed, unfused, flags=fl, **kw)
        return r
    g, plan, inputs, dev = prepare(spec, seed, **kw)
    for info in plan.groups:
        assert info.status == 0, info
    outs = [info.out for info in plan.groups]
    ref = OE.run_unfused(spec, inputs, keep=outs)
    env = run_fused(plan, spec, dev)
    plan.sync()
    worst = 0.0
    for vid in outs:
        worst = max(worst, check_parity(spec, vid, env[vid].cpu().numpy(), ref[vid]))
    if unfused:
        envu = run_unfused(plan, spec, dev)
        plan.sync()
        for vid in spec.outputs:
            check_parity(spec, vid, envu[vid].cpu().numpy(), ref[vid])
    return plan, env, ref, worst


@pytest.mark.parametrize("shape", [(200, 132), (64, 64), (33, 96), (1, 256), (96, 4), (4, 8)])
def test_diamond_small_shapes(shape):
    plan, env, ref, _ = _check(W.diamond(*shape))
    assert plan.n_groups == 1


def test_diamond_full_size():
    spec = W.diamond(8192, 4096)
    g, plan, inputs, dev = prepare(spec)
    env = run_fused(plan, spec, dev)
    plan.sync()
    out = env[spec.outputs[0]].cpu().numpy()
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    assert rel_err(out, ref) <= TOL_F32


def test_diamond_odd_width_uses_direct_paths():
    """A frame width that is not a multiple of 4 floats cannot use TMA: the
    plan gathers those leaves and stores directly."""
    spec = W.diamond(37, 30)
    plan, *_ = _check(spec)
    assert plan.exec_info(0)["n_gathered"] >= 1


@pytest.mark.parametrize("epi", [False, True])
def test_rnnlm_chain(epi):
    plan, env, ref, _ = _check(W.rnnlm_chain(), allow_reduce_epilogue=epi)
    assert plan.n_groups == (1 if epi else 2)


@pytest.mark.parametrize("epi", [False, True])
def test_rnnlm_chain_scaled(epi):
    # the bandwidth-bound variant of the chain: X, Y [65536, 1024] (512 MiB)
    plan, env, ref, _ = _check(W.rnnlm_chain(65536, 1024), unfused=False, allow_reduce_epilogue=epi, flags=0)
    assert plan.n_groups == (1 if epi else 2)


@pytest.mark.parametrize("shape", [(64, 1024), (100, 200), (8192, 4096), (4096, 8192), (3, 2052)])
def test_row_reductions(shape):
    R, C = shape
    for op in ("rowsum", "rowmax"):
        spec = W.GraphSpec()
        x = spec.input((R, C))
        y = spec.input((R, C))
        v = spec.input((C,))
        a = spec.op("mul", (x, y))
        b = spec.op("badd_col", (a, v))
        s = spec.op(op, (b,))
        spec.mark_output(s)
        assert exact_value(spec, s) == (op == "rowmax")
        _check(spec, unfused=(R * C <= 1 << 20))


def test_reduce_of_transposed_operand():
    spec = W.GraphSpec()
    x = spec.input((96, 160))
    t = spec.op("transpose", (x,))
    r = spec.op("tanh", (t,))
    y = spec.input((160, 96))
    a = spec.op("add", (r, y))
    s = spec.op("rowsum", (a,))
    spec.mark_output(s)
    _check(spec)


def test_all_elementwise_ops():
    spec = W.GraphSpec()
    x = spec.input((64, 96))
    y = spec.input((64, 96), init=("uniform", 0.5, 2.0))
    vr = spec.input((64,))
    vc = spec.input((96,))
    a = spec.op("sub", (x, y))
    b = spec.op("div", (a, y))
    c = spec.op("addc", (b,), (0.25,))
    d = spec.op("neg", (c,))
    e = spec.op("sigmoid", (d,))
    f = spec.op("bmul_row", (e, vr))
    h = spec.op("badd_row", (f, vr))
    i = spec.op("bmul_col", (h, vc))
    j = spec.op("tanh", (i,))
    k = spec.op("exp", (j,))
    spec.mark_output(k)
    plan, *_ = _check(spec)
    assert plan.n_groups == 1


@pytest.mark.parametrize("shape", [(64, 32), (4096, 8192), (37, 30), (1, 4), (2, 4)])
def test_injective_only_groups(shape):
    """Groups of transposes and reshapes alone (index maps, no arithmetic):
    every output bit for bit equal to the oracle's, staged and gathered.  A
    reshape of a transposed value whose digits do not split at a row boundary
    is refused by the plan, so the chain runs on power-of-two shapes."""
    R, C = shape
    spec = W.GraphSpec()
    x = spec.input((R, C))
    spec.mark_output(spec.op("transpose", (x,)))
    specs = [spec]
    if R & (R - 1) == 0 and C & (C - 1) == 0:
        spec2 = W.GraphSpec()
        y = spec2.input((R, C))
        t = spec2.op("transpose", (y,))                 # [C, R]
        r = spec2.op("reshape", (t,), (R, C))           # reinterpret
        u = spec2.op("transpose", (r,))                 # [C, R]
        spec2.mark_output(spec2.op("reshape", (u,), (2 * R, C // 2)))
        specs.append(spec2)
    for sp in specs:
        assert exact_value(sp, sp.outputs[0])
        plan, *_ = _check(sp, unfused=(R * C <= 1 << 20))
        assert plan.n_groups == 1


def test_transpose_reshape_chains():
    """Leaves read through composed transposes and reshapes (digit maps)."""
    spec = W.GraphSpec()
    x = spec.input((64, 32))
    t = spec.op("transpose", (x,))            # [32, 64]
    r = spec.op("reshape", (t,), (64, 32))    # reinterpret
    y = spec.input((64, 32))
    a = spec.op("add", (r, y))
    u = spec.op("transpose", (a,))            # [32, 64]
    w = spec.op("relu", (u,))
    spec.mark_output(w)
    plan, *_ = _check(spec)
    assert plan.n_groups == 1


@pytest.mark.parametrize("seed", range(6))
def test_random_dag_small(seed):
    spec = W.random_dag(seed, **W.CONFIGS["random_dag"]["small"])
    _check(spec, seed=seed)


def test_random_dag_full_size():
    """The random DAG at its full size (seed 0: 200 operators over [8192, 4096]
    and [4096, 8192] values), partitioned and launched as the benchmark runs
    it: every graph output against the oracle (about a minute of host time)."""
    spec = W.random_dag(0)
    g, plan, inputs, dev = prepare(spec, 0)
    for info in plan.groups:
        assert info.status == 0, info
    ref = OE.run_unfused(spec, inputs)
    env = run_fused(plan, spec, dev)
    plan.sync()
    assert len(spec.outputs) > 10
    for vid in spec.outputs:
        check_parity(spec, vid, env[vid].cpu().numpy(), ref[vid])


def test_launch_rejects_bad_pointers():
    from group_execution_gb300 import FgError
    spec = W.diamond(64, 32)
    g, plan, inputs, dev = prepare(spec)
    info = plan.groups[0]
    out = torch.empty((32, 64), device="cuda")
    ptrs = {v: dev[v] for v in info.leaves}
    ptrs[info.out] = out
    ptrs[info.leaves[0]] = dev[info.leaves[0]].data_ptr() + 4      # misaligned
    with pytest.raises(FgError):
        plan.launch_group(0, ptrs)
    ptrs[info.leaves[0]] = 0
    with pytest.raises(FgError):
        plan.launch_group(0, ptrs)
    plan.launch_group(0, {v: dev[v] for v in info.leaves} | {info.out: out})
    plan.sync()


@pytest.mark.parametrize("tpu", [1, 2, 5, 16])
@pytest.mark.parametrize("shape", [(1024, 4096), (700, 1000)])
def test_row_reductions_forced_splits(tpu, shape):
    """Rows cut into units of `tpu` column tiles (flag bits 16-23): many split
    units per CTA, so every consumer warp in turn publishes partials and
    finishes strips across consecutive units; with an epilogue on the reduced
    vector; run twice (the strips' counters are cleared by their finishers)."""
    R, C = shape
    for op in ("rowsum", "rowmax"):
        for epi in (True, False):
            spec = W.GraphSpec()
            x = spec.input((R, C))
            v = spec.input((C,))
            s = spec.op(op, (spec.op("badd_col", (spec.op("relu", (x,)), v)),))
            spec.mark_output(spec.op("sigmoid", (s,)) if epi else s)
            out = spec.outputs[0]
            # a maximum without the sigmoid epilogue is compared bit for bit
            assert exact_value(spec, out) == (op == "rowmax" and not epi)
            g, plan, inputs, dev = prepare(spec, 0, allow_reduce_epilogue=epi, flags=tpu << 16)
            assert plan.n_groups == 1 and plan.groups[0].kind == "reduce"
            ref = OE.run_unfused(spec, inputs)[out]
            for _ in range(2):
                env = run_fused(plan, spec, dev)
                plan.sync()
                check_parity(spec, out, env[out].cpu().numpy(), ref)


def test_small_groups_get_the_direct_kernel():
    """Groups of at most 2 MiB carry the small-group kernel; larger ones,
    groups built with flag bit 28 and interpreted groups do not."""
    small = graph_from_spec(W.rnnlm_chain()).build(allow_reduce_epilogue=True)
    assert "fg_jit_small_group" in small.source(0)
    big = graph_from_spec(W.diamond(1024, 1024)).build()
    assert "fg_jit_small_group" not in big.source(0)
    off = graph_from_spec(W.rnnlm_chain()).build(allow_reduce_epilogue=True, flags=_lib.FG_FLAG_NO_SMALL)
    assert "fg_jit_small_group" not in off.source(0)


@pytest.mark.parametrize("shape", [(64, 1024), (37, 30), (1, 4), (300, 1000), (5, 2100)])
@pytest.mark.parametrize("op", ["rowsum", "rowmax"])
def test_small_kernel_reductions_both_paths(shape, op):
    """A reduce group with a broadcast prologue and an epilogue, small enough
    for the direct kernel, against the oracle on both paths."""
    R, C = shape
    spec = W.GraphSpec()
    x = spec.input((R, C))
    v = spec.input((C,))
    s = spec.op(op, (spec.op("badd_col", (spec.op("relu", (x,)), v)),))
    spec.mark_output(spec.op("sigmoid", (s,)))
    for fl in (0, _lib.FG_FLAG_NO_SMALL):
        _check(spec, allow_reduce_epilogue=True, flags=fl)


@pytest.mark.parametrize("shape", [(1, 1), (1, 3), (5, 1), (2, 1), (4096, 1), (1, 1025), (3, 2)])
def test_degenerate_frames(shape):
    """Single-element, single-row and single-column frames: the diamond
    group (its transposed output of a single column is a reinterpretation,
    so the leaves are read in place) and a row reduction with a broadcast
    prologue and an epilogue, each through the direct kernel, the pipeline
    and the interpreter, fused and unfused; maxima bit for bit."""
    _check(W.diamond(*shape))
    R, C = shape
    for op in ("rowsum", "rowmax"):
        spec = W.GraphSpec()
        x = spec.input((R, C))
        v = spec.input((C,))
        s = spec.op(op, (spec.op("badd_col", (spec.op("relu", (x,)), v)),))
        spec.mark_output(s)
        plan, env, ref, _ = _check(spec)
        if op == "rowmax":
            assert exact_value(spec, s)
            np.testing.assert_array_equal(env[s].cpu().numpy(), ref[s])
