"""GPU parity of the direct kernel on large row reductions (one warp per frame
row segment, leaves read straight from global memory) against the CPU
oracle, through the C ABI.  The shapes split rows into 4, 2 and 1 segments,
with ragged last segments and widths whose last pass is shorter than a lane's
eight columns; the programs read the frame's own layout, a vector over its
columns and a vector over its rows, and one applies an epilogue to the
reduced vector.  Results computed by exact operators alone (row maxima of
sums and products) must match bit for bit; row sums within the float32
tolerance.  The same plans built without the direct kernel (flag bit 28)
must match as well."""
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import execute as OE
from tests._helpers import check_parity
from tests._gpu import prepare, run_fused
from group_execution_gb300 import _lib

pytestmark = pytest.mark.gpu

# (shape, warps per row)
SHAPES = [((8192, 4096), 4), ((2048, 4100), 4), ((4096, 2052), 2), ((8192, 1028), 1)]


def _sum(R, C):
    g = W.GraphSpec("rowsum")
    g.mark_output(g.op("rowsum", (g.input((R, C)),)))
    return g


def _max_row_vector(R, C):
    g = W.GraphSpec("rowmax_badd_row")
    x, r = g.input((R, C)), g.input((R,))
    g.mark_output(g.op("rowmax", (g.op("badd_row", (x, r)),)))
    return g


def _max_products(R, C):
    g = W.GraphSpec("rowmax_mul_bmul_col")
    x, y, w = g.input((R, C)), g.input((R, C)), g.input((C,))
    g.mark_output(g.op("rowmax", (g.op("bmul_col", (g.op("mul", (x, y)), w)),)))
    return g


PROGRAMS = {"rowsum": (_sum, False), "rowmax_row_vector": (_max_row_vector, False),
            "rowmax_products": (_max_products, False), "rnnlm_epilogue": (W.rnnlm_chain, True)}


@pytest.mark.parametrize("shape,seg", SHAPES, ids=[f"{s[0]}x{s[1]}" for s, _ in SHAPES])
@pytest.mark.parametrize("prog", list(PROGRAMS))
@pytest.mark.parametrize("direct", [True, False])
def test_direct_row_reduction(shape, seg, prog, direct):
    make, epi = PROGRAMS[prog]
    spec = make(*shape)
    flags = 0 if direct else _lib.FG_FLAG_NO_SMALL
    g, plan, inputs, dev = prepare(spec, seed=sum(shape), flags=flags, allow_reduce_epilogue=epi)
    assert plan.n_groups == 1
    info = plan.direct_info(0)
    assert info["direct"] == (1 if direct else 0)
    if direct:
        assert info["segments"] == seg
    env = run_fused(plan, spec, dev)
    plan.sync()
    out = spec.outputs[0]
    ref = OE.run_unfused(spec, inputs)[out]
    check_parity(spec, out, env[out].cpu().numpy(), ref)


def test_direct_after_pipelined_and_back():
    """Launch order does not change results: a large direct reduction behind a
    pipelined group (launched without early start) and behind another direct
    launch (launched early) on one stream."""
    spec = W.rnnlm_chain(8192, 4096)
    g, plan, inputs, dev = prepare(spec, seed=5)
    assert plan.n_groups == 2 and plan.direct_info(0)["direct"] == 1
    assert plan.direct_info(0)["early_launch"] == 0
    ref = OE.run_unfused(spec, inputs, keep=[gi.out for gi in plan.groups])
    env = dict(dev)
    for v in spec.ops:
        env[v.vid] = torch.empty(v.shape, device="cuda")
    ptrs = [{v: env[v] for v in gi.leaves + gi.outs} for gi in plan.groups]
    for _ in range(2):
        plan.launch_group(0, ptrs[0])
        plan.launch_group(0, ptrs[0])   # behind a direct launch: starts early
        plan.launch_group(1, ptrs[1])
    plan.sync()
    for gi in plan.groups:
        check_parity(spec, gi.out, env[gi.out].cpu().numpy(), ref[gi.out])
