"""Host logic of the direct kernel's choice (no device needed): which groups
fg_launch_group runs on it, with how many warps per frame row, and whether
their launch always may start early."""
import pytest

import workloads as W
from group_execution_gb300 import _lib, graph_from_spec


def _rowsum(R, C):
    g = W.GraphSpec("rowsum")
    g.mark_output(g.op("rowsum", (g.input((R, C)),)))
    return g


# (shape, direct, segments): row reductions of at least 8192 row segments
# (rows x warps per row) with every leaf read row by row; widths that are
# not a multiple of 4 floats make their leaves gathers (pipeline); small
# groups with rows of at most 1024 columns always go direct
CASES = [((8192, 4096), 1, 4), ((4096, 8192), 1, 4), ((2048, 4100), 1, 4), ((2047, 4096), 0, 1),
         ((4096, 2052), 1, 2), ((4095, 2048), 0, 1), ((8192, 1028), 1, 1), ((8191, 1024), 0, 1),
         ((65536, 512), 0, 1), ((2048, 4097), 0, 1), ((64, 1024), 1, 1), ((1, 65536), 0, 1)]


@pytest.mark.parametrize("shape,direct,seg", CASES, ids=[f"{s[0]}x{s[1]}" for s, _, _ in CASES])
def test_direct_choice(shape, direct, seg):
    plan = graph_from_spec(_rowsum(*shape)).build()
    info = plan.direct_info(0)
    assert (info["direct"], info["segments"]) == (direct, seg)
    # a large direct launch starts early only behind another direct launch;
    # small groups always may
    small = shape[0] * shape[1] * 4 <= (2 << 20) and shape[1] <= 1024
    assert info["early_launch"] == (1 if small or not direct else 0)


def test_direct_off_by_flag_and_for_transposed_leaves():
    plan = graph_from_spec(_rowsum(8192, 4096)).build(flags=_lib.FG_FLAG_NO_SMALL)
    assert plan.direct_info(0) == {"direct": 0, "segments": 1, "early_launch": 1}
    # a row sum of a transposed value reads its leaf column by column
    g = W.GraphSpec("rowsum_t")
    x = g.input((4096, 8192))
    g.mark_output(g.op("rowsum", (g.op("transpose", (x,)),)))
    plan = graph_from_spec(g).build()
    assert plan.direct_info(0)["direct"] == 0


def test_elementwise_groups_use_one_segment():
    plan = graph_from_spec(W.rnnlm_chain()).build()
    for gid in range(plan.n_groups):
        info = plan.direct_info(gid)
        assert info["direct"] == 1 and info["segments"] == 1 and info["early_launch"] == 1
    plan = graph_from_spec(W.diamond(8192, 4096)).build()
    assert plan.direct_info(0)["direct"] == 0


def test_direct_info_errors():
    plan = graph_from_spec(_rowsum(64, 64)).build()
    with pytest.raises(_lib.FgError):
        plan.direct_info(1)
