"""Host checks of the largest and the degenerate extents (no device needed):
graph inputs take extents from 1 to 2^31 - 64 per axis and refuse the rest;
a frame of 2^31 or more elements builds when every leaf is staged through TMA
(whose coordinates are per axis) and its group reports FG_EUNSUPPORTED when a
leaf would have to be gathered (gathers index the frame with 32-bit flat
offsets); a single-element frame and a single-row frame build like any
other."""
import ctypes as C

import pytest

from group_execution_gb300 import Graph, _lib

BIG = (1 << 31) - 64


def _add_input(shape):
    g = Graph()
    lib = _lib.load()
    vid = C.c_int32()
    shp = (C.c_int64 * len(shape))(*shape)
    return lib.fg_graph_add_input(g.h, _lib.FG_F32, len(shape), shp, C.byref(vid)), g


@pytest.mark.parametrize("shape", [(0,), (0, 4), (4, 0), (-1, 4), (4, -8), (BIG + 1, 1), (1, BIG + 1)])
def test_extents_refused(shape):
    st, _ = _add_input(shape)
    assert st == _lib.FG_ESHAPE


@pytest.mark.parametrize("shape", [(1,), (1, 1), (BIG, 1), (1, BIG), (BIG,), (65536, 65536)])
def test_extents_accepted(shape):
    st, _ = _add_input(shape)
    assert st == _lib.FG_OK


def _relu_group(R, Cc):
    g = Graph()
    x = g.input((R, Cc))
    g.mark_output(g.op("relu", (x,)))
    return g.build()


def test_frame_of_2_pow_31_elements_with_staged_leaves():
    # 2^31 elements, a width of whole 16-byte rows: the leaf is staged
    plan = _relu_group(1 << 16, 1 << 15)
    assert plan.n_groups == 1 and plan.groups[0].status == _lib.FG_OK
    info = plan.exec_info(0)
    assert info["n_staged"] == 1 and info["n_gathered"] == 0
    assert plan.groups[0].alg_bytes == 2 * (1 << 31) * 4


def test_frame_of_2_pow_31_elements_with_a_gathered_leaf():
    # 524288 x 4099 = 2,149,056,512 > 2^31: rows of 4099 floats are not
    # 16-byte multiples, so the leaf would be gathered with 32-bit offsets
    plan = _relu_group(1 << 19, 4099)
    assert plan.n_groups == 1 and plan.groups[0].status == _lib.FG_EUNSUPPORTED
    lib = _lib.load()
    assert lib.fg_plan_group_info(plan.h, 0, None, None, None, None, None, None, None, None) == _lib.FG_EUNSUPPORTED
    assert b"2^31" in lib.fg_last_error()
    # the launch is refused before any pointer or device is looked at
    assert lib.fg_launch_group(plan.h, 0, None, None) == _lib.FG_EUNSUPPORTED


def test_gathered_leaf_just_below_2_pow_31():
    # 523,900 x 4099 = 2,147,466,100 < 2^31: gathering is exact there
    plan = _relu_group(523_900, 4099)
    assert plan.groups[0].status == _lib.FG_OK
    info = plan.exec_info(0)
    assert info["n_gathered"] == 1 and info["n_staged"] == 0


@pytest.mark.parametrize("shape", [(1, 1), (1, 4096), (4096, 1), (1, 3)])
def test_degenerate_frames_build(shape):
    g = Graph()
    x, y = g.input(shape), g.input(shape)
    s = g.op("add", (g.op("relu", (x,)), y))
    g.mark_output(g.op("rowsum", (s,)))
    plan = g.build()
    assert plan.n_groups == 1
    assert plan.groups[0].alg_bytes == (2 * shape[0] * shape[1] + shape[0]) * 4
