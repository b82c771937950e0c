"""Random, mostly malformed, graph-building calls through the C ABI (no GPU
needed): bad opcodes, arities, value ids, attributes, dtypes and shapes must
come back as error statuses, never a crash, and whatever graph results must
build (or be refused) with consistent queries.  The same calls were also run
against a build of the host sources with -fsanitize=address,undefined."""
import ctypes as C

import numpy as np
import pytest

from group_execution_gb300 import _lib

STATUSES = {_lib.FG_OK, _lib.FG_EINVAL, _lib.FG_ESHAPE, _lib.FG_EUNSUPPORTED}
DIMS = [1, 2, 3, 4, 8, 16, 24, 32, 48, 64, 0, -1, 5]


def _random_graph(lib, r):
    g = C.c_void_p()
    assert lib.fg_graph_create(C.byref(g)) == _lib.FG_OK
    nvals = 0
    for _ in range(int(r.integers(1, 40))):
        vid = C.c_int32(-7)
        if nvals == 0 or r.random() < 0.3:
            shape = (C.c_int64 * 4)(*[int(r.choice(DIMS)) for _ in range(4)])
            st = lib.fg_graph_add_input(g, int(r.choice([0, 0, 1, 2, -1])), int(r.choice([1, 2, 2, 2, 0, 3])),
                                        shape, C.byref(vid))
        else:
            nin = int(r.choice([0, 1, 2, 3, 4, 1, 2]))
            ins = (C.c_int32 * max(nin, 1))(*[int(r.integers(-1, nvals + 1)) if r.random() < 0.1
                                              else int(r.integers(0, nvals)) for _ in range(max(nin, 1))])
            nat = int(r.choice([0, 0, 1, 2, 3]))
            at = (C.c_float * 3)(*[float(r.choice([0.5, 2.0, 1.0, 0.0, -1.0, 16, 8, 4, 64, np.nan]))
                                   for _ in range(3)])
            st = lib.fg_graph_add_op(g, int(r.integers(-1, len(_lib.OPCODES) + 1)), nin, ins if nin else None,
                                     nat, at if nat else None, C.byref(vid))
        assert st in STATUSES
        if st == _lib.FG_OK:
            assert vid.value == nvals
            nvals += 1
        if nvals and r.random() < 0.15:
            assert lib.fg_graph_mark_output(g, int(r.integers(-1, nvals + 1))) in STATUSES
    return g


def _check_plan(lib, p):
    nn, ng = C.c_int32(), C.c_int32()
    assert lib.fg_plan_query(p, C.byref(nn), C.byref(ng), None, None) == _lib.FG_OK
    go, ip = (C.c_int32 * max(nn.value, 1))(), (C.c_int32 * max(nn.value, 1))()
    assert lib.fg_plan_query(p, C.byref(nn), C.byref(ng), go, ip) == _lib.FG_OK
    assert 1 <= ng.value <= nn.value
    assert all(-1 <= ip[i] < nn.value for i in range(nn.value))
    assert all(i <= go[i] < nn.value for i in range(nn.value))      # a group is labelled by its sink
    covered = 0
    for gid in range(-1, ng.value + 1):
        n_nodes, n_leaves, out, kind = C.c_int32(), C.c_int32(), C.c_int32(), C.c_int32()
        ab, af = C.c_int64(), C.c_int64()
        st = lib.fg_plan_group_info(p, gid, C.byref(n_nodes), None, C.byref(n_leaves), None, C.byref(out),
                                    C.byref(kind), C.byref(ab), C.byref(af))
        if not 0 <= gid < ng.value:
            assert st == _lib.FG_EINVAL
            continue
        # a group the kernels cannot run keeps its grouping and says so
        assert st in (_lib.FG_OK, _lib.FG_EUNSUPPORTED)
        covered += n_nodes.value
        nodes = (C.c_int32 * n_nodes.value)()
        leaves = (C.c_int32 * max(n_leaves.value, 1))()
        assert lib.fg_plan_group_info(p, gid, C.byref(n_nodes), nodes, C.byref(n_leaves), leaves, C.byref(out),
                                      C.byref(kind), C.byref(ab), C.byref(af)) == st
        sink = max(nodes)
        assert all(go[x] == sink for x in nodes)
        if st == _lib.FG_OK:
            n = C.c_int64()
            assert lib.fg_plan_group_source(p, gid, None, 0, C.byref(n)) == _lib.FG_OK
            buf = C.create_string_buffer(17)             # a short buffer is truncated, not overrun
            assert lib.fg_plan_group_source(p, gid, buf, 17, C.byref(n)) == _lib.FG_OK
            assert len(buf.value) <= 16
    assert covered == nn.value


@pytest.mark.parametrize("block", range(8))
def test_random_graph_calls(block):
    lib = _lib.load()
    plans = 0
    for seed in range(block * 250, (block + 1) * 250):
        r = np.random.default_rng(seed)
        g = _random_graph(lib, r)
        opts = _lib.BuildOpts()
        lib.fg_build_opts_default(C.byref(opts))
        opts.max_fused_ops = int(r.choice([256, 1, 2, 3]))
        opts.max_args = int(r.choice([64, 1, 2, 3, 4]))
        opts.allow_reduce_epilogue = int(r.integers(0, 2))
        p = C.c_void_p()
        st = lib.fg_build_groups(g, C.byref(opts), C.byref(p))
        assert st in STATUSES
        if st == _lib.FG_OK:
            plans += 1
            _check_plan(lib, p)
            lib.fg_plan_destroy(p)
        lib.fg_graph_destroy(g)
    assert plans > 50
