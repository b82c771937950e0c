"""GPU parity of groups holding tuples and concatenations (TVM "Operator
Fusion": a tuple fuses into the injective op after it in phase 1, its fields'
producers join in phase 2): every value a group writes, against the oracle,
through the C ABI, compiled programs."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import execute as OE
from oracle import partition as OP
from tests._helpers import check_parity, exact_value, tuple_dag
from tests._gpu import prepare, run_fused, run_unfused

pytestmark = pytest.mark.gpu


def _check(spec, seed=0, unfused=True):
    g, plan, inputs, dev = prepare(spec, seed)
    assert plan.group_of == OP.partition(spec)[0]
    for info in plan.groups:
        assert info.status == 0, info
    ref = OE.run_unfused(spec, inputs, keep=[v.vid for v in spec.ops])
    env = run_fused(plan, spec, dev)
    plan.sync()
    for info in plan.groups:
        for o in info.outs:
            check_parity(spec, o, env[o].cpu().numpy(), ref[o])
    if unfused:
        envu = run_unfused(plan, spec, dev)
        plan.sync()
        for o in spec.outputs:
            check_parity(spec, o, envu[o].cpu().numpy(), ref[o])
    return plan


def _inception(r1, r2, C, transpose=False, three=False):
    g = W.GraphSpec()
    a = g.op("relu", (g.input((r1, C)),))
    b = g.op("exp", (g.input((r2, C)),))
    fields = [a, b]
    if three:
        fields.append(g.op("transpose", (g.input((C, 16)),)))
    c = g.op("concat", (g.op("tuple", tuple(fields)),))
    if transpose:
        c = g.op("transpose", (c,))
    g.mark_output(g.op("scale", (c,), (0.5,)))
    return g


@pytest.mark.parametrize("r1,r2,C", [(64, 32, 64), (40, 24, 32), (37, 29, 20), (300, 212, 96)])
@pytest.mark.parametrize("transpose", [False, True])
def test_concat_only_bit_exact(r1, r2, C, transpose):
    """A tuple of inputs concatenated (and transposed): an injective-only
    group, equal to the oracle bit for bit."""
    g = W.GraphSpec()
    c = g.op("concat", (g.op("tuple", (g.input((r1, C)), g.input((r2, C)))),))
    if transpose:
        c = g.op("transpose", (c,))
    g.mark_output(c)
    assert exact_value(g, c)
    plan = _check(g)
    assert plan.n_groups == 1


@pytest.mark.parametrize("r1,r2,C", [(64, 32, 64), (40, 24, 32), (37, 29, 20), (300, 212, 96)])
@pytest.mark.parametrize("transpose", [False, True])
def test_inception(r1, r2, C, transpose):
    plan = _check(_inception(r1, r2, C, transpose))
    assert plan.n_groups == 1


def test_three_fields_with_a_transposed_one():
    plan = _check(_inception(48, 33, 64, three=True))
    assert plan.n_groups == 1


def test_full_size_inception():
    plan = _check(_inception(4096, 4096, 4096), unfused=False)
    assert plan.n_groups == 1


@pytest.mark.parametrize("seed", range(12))
def test_random_tuple_graphs(seed):
    _check(tuple_dag(seed), seed)
