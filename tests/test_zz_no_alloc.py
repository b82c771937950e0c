"""The row reduction that allocates no device memory.

It exists for callers that cannot call cudaMalloc (a framework that owns all
device allocations through its own pool, or a step that cannot accept an
allocation's implicit synchronisation): its scratch lives in a fixed device
array instead of plan-owned memory.  Its results must match the plan-based
reduce group (the existing entry point, fg_launch_group) within the float32
tolerance, on two calls in a row, since every call reuses the same scratch.
This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from group_execution_gb300 import _lib, graph_from_spec
from tests._helpers import rel_err, TOL_F32

pytestmark = pytest.mark.gpu

OPS = {"rowsum": 17, "rowmax": 18}


def _plan_reference(op, x):
    spec = W.GraphSpec()
    vx = spec.input(tuple(x.shape))
    vy = spec.op(op, (vx,))
    spec.mark_output(vy)
    plan = graph_from_spec(spec).build()
    y = torch.empty((x.shape[0],), device="cuda")
    plan.launch_group(0, {vx: x, vy: y})
    plan.sync()
    return y.cpu().numpy()


def _noalloc(lib, op, x, y):
    st = lib.fg_row_reduce_noalloc(OPS[op], C.c_void_p(x.data_ptr()), x.shape[0], x.shape[1],
                                   C.c_void_p(y.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.fg_last_error()


@pytest.mark.parametrize("shape", [(8192, 4096), (4096, 8192), (100, 200), (3, 2052), (65536, 64), (37, 30)])
@pytest.mark.parametrize("op", ["rowsum", "rowmax"])
def test_noalloc_matches_plan_two_calls(shape, op):
    lib = _lib.load()
    rng = np.random.default_rng(hash((shape, op)) % 2 ** 32)
    x = torch.from_numpy(rng.uniform(-1, 1, size=shape).astype(np.float32)).cuda()
    ref = _plan_reference(op, x)
    for _ in range(2):
        y = torch.full((shape[0],), float("nan"), device="cuda")
        _noalloc(lib, op, x, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        if op == "rowmax":
            np.testing.assert_array_equal(got, ref)


def test_noalloc_rejects_oversize_and_bad_args():
    lib = _lib.load()
    x = torch.zeros((65537, 4), device="cuda")
    y = torch.zeros((65537,), device="cuda")
    s = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fg_row_reduce_noalloc(17, C.c_void_p(x.data_ptr()), 65537, 4, C.c_void_p(y.data_ptr()), s) \
        == _lib.FG_EINVAL
    assert b"65536" in lib.fg_last_error()
    assert lib.fg_row_reduce_noalloc(3, C.c_void_p(x.data_ptr()), 4, 4, C.c_void_p(y.data_ptr()), s) \
        == _lib.FG_EINVAL
    assert lib.fg_row_reduce_noalloc(17, None, 4, 4, C.c_void_p(y.data_ptr()), s) == _lib.FG_EINVAL
