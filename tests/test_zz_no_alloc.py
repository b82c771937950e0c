"""The row reduction that allocates no device memory.

It exists for callers that cannot call cudaMalloc (a framework that owns all
device allocations through its own pool, or a step that cannot accept an
allocation's implicit synchronisation): its scratch lives in a fixed device
array instead of plan-owned memory.  Its results must match the oracle's row
sum (float32 tolerance) and row maximum (bit for bit), and the plan-based
reduce group (the existing entry point, fg_launch_group) within the same
tolerance, on two calls in a row, since every call reuses the same scratch.
The shapes cover the staged path (columns a multiple of 4) and the gathered
one, each with and without column splits.  After a warm-up call, further
calls must leave the device's free memory unchanged, and the error word must
read clear.  This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from group_execution_gb300 import _lib, graph_from_spec
from oracle import execute as OE
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


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(lib, op, x, y):
    st = lib.fg_row_reduce_noalloc(OPS[op], C.c_void_p(x.data_ptr()), x.shape[0], x.shape[1],
                                   C.c_void_p(y.data_ptr()), _stream())
    assert st == 0, lib.fg_last_error()


# (8192, 4096), (4096, 8192), (65536, 64): staged rows, one split per strip or
# several; (100, 200), (3, 2052): staged, ragged tails; (37, 30): gathered, one
# split; (256, 4097), (40, 8191): gathered rows cut into several column splits
SHAPES = [(8192, 4096), (4096, 8192), (100, 200), (3, 2052), (65536, 64), (37, 30), (256, 4097), (40, 8191)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("op", ["rowsum", "rowmax"])
def test_noalloc_matches_oracle_and_plan_two_calls(shape, op):
    lib = _lib.load()
    rng = np.random.default_rng([shape[0], shape[1], OPS[op]])
    xh = rng.uniform(-1, 1, size=shape).astype(np.float32)
    x = torch.from_numpy(xh).cuda()
    ref = OE.apply_op(op, [xh], ())
    plan_ref = _plan_reference(op, x)
    for _ in range(2):
        y = torch.full((shape[0],), float("nan"), device="cuda")
        _noalloc(lib, op, x, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(got, plan_ref) <= TOL_F32
        if op == "rowmax":
            np.testing.assert_array_equal(got, ref)
    assert lib.fg_row_reduce_noalloc_status(_stream()) == _lib.FG_OK, lib.fg_last_error()


def test_noalloc_allocates_nothing():
    """Once each path has run (loading the module and its kernels), more calls
    leave the device's free memory exactly as it was."""
    lib = _lib.load()
    xs = [torch.rand((4096, 4096), device="cuda"), torch.rand((256, 4097), device="cuda")]
    ys = [torch.empty((x.shape[0],), device="cuda") for x in xs]
    for x, y in zip(xs, ys):
        for op in OPS:
            _noalloc(lib, op, x, y)
    assert lib.fg_row_reduce_noalloc_status(_stream()) == _lib.FG_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(10):
        for x, y in zip(xs, ys):
            for op in OPS:
                _noalloc(lib, op, x, y)
    assert lib.fg_row_reduce_noalloc_status(_stream()) == _lib.FG_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_oversize_and_bad_args():
    lib = _lib.load()
    x = torch.zeros((65537, 4), device="cuda")
    y = torch.zeros((65537,), device="cuda")
    s = _stream()
    assert lib.fg_row_reduce_noalloc(17, C.c_void_p(x.data_ptr()), 65537, 4, C.c_void_p(y.data_ptr()), s) \
        == _lib.FG_EINVAL
    assert b"65536" in lib.fg_last_error()
    assert lib.fg_row_reduce_noalloc(3, C.c_void_p(x.data_ptr()), 4, 4, C.c_void_p(y.data_ptr()), s) \
        == _lib.FG_EINVAL
    assert lib.fg_row_reduce_noalloc(17, None, 4, 4, C.c_void_p(y.data_ptr()), s) == _lib.FG_EINVAL
