"""Failure detection without a GPU fault: with the failure-injection hook the
kernels' load producers issue nothing, so every consumer's bounded wait
(1 ms here) expires.  The kernel records FG_ETIMEOUT in the plan's device
flag and returns; fg_sync_status reports it, clears it, and the context stays
usable for a correct run right after."""
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import execute as OE
from tests._helpers import rel_err, TOL_F32
from tests._gpu import prepare, run_fused
from group_execution_gb300 import _lib, FgError

pytestmark = pytest.mark.gpu
MODES = [0, _lib.FG_FLAG_INTERPRET]


def _spec(case):
    if case == "elementwise":
        return W.diamond(256, 128)
    if case == "reduce":
        return W.rnnlm_chain()
    return W.sf_update(128, 256, 512)


@pytest.mark.parametrize("case", ["elementwise", "reduce", "gemm"])
@pytest.mark.parametrize("mode", MODES)
def test_injected_timeout_is_reported_and_recoverable(case, mode):
    spec = _spec(case)
    g, plan, inputs, dev = prepare(spec, flags=mode | _lib.FG_FLAG_INJECT_NO_LOADS, wait_limit_ns=1_000_000)
    run_fused(plan, spec, dev)
    with pytest.raises(FgError) as e:
        plan.sync()
    assert e.value.status == _lib.FG_ETIMEOUT
    plan.sync()                       # the flag was cleared
    # same process, same context: a normal plan still runs correctly
    g2, plan2, inputs2, dev2 = prepare(spec, flags=mode)
    env = run_fused(plan2, spec, dev2)
    plan2.sync()
    ref = OE.run_unfused(spec, inputs2)
    for o in spec.outputs:
        assert rel_err(env[o].cpu().numpy(), ref[o]) <= TOL_F32

