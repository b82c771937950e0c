"""The compiled group programs (straight-line CUDA generated per group) are
valid sm_103a code: NVRTC compiles them on the host, without a GPU."""
import pytest

import workloads as W
from group_execution_gb300 import graph_from_spec

nvrtc = pytest.importorskip("cuda.bindings.nvrtc")


def _compile(src):
    err, prog = nvrtc.nvrtcCreateProgram(src.encode(), b"group.cu", 0, [], [])
    assert err == nvrtc.nvrtcResult.NVRTC_SUCCESS
    opts = [b"--gpu-architecture=sm_103a", b"--std=c++17"]
    (rc,) = nvrtc.nvrtcCompileProgram(prog, len(opts), opts)
    _, n = nvrtc.nvrtcGetProgramLogSize(prog)
    log = b" " * n
    nvrtc.nvrtcGetProgramLog(prog, log)
    nvrtc.nvrtcDestroyProgram(prog)
    assert rc == nvrtc.nvrtcResult.NVRTC_SUCCESS, log.decode()[:3000]


@pytest.mark.parametrize("name,kw", [("diamond", {}), ("rnnlm_chain", {"allow_reduce_epilogue": True}),
                                     ("rnnlm_chain", {}), ("sf_update", {})])
def test_config_programs_compile(name, kw):
    spec = getattr(W, name)(**W.CONFIGS[name]["small"])
    plan = graph_from_spec(spec).build(**kw)
    for gid in range(plan.n_groups):
        src = plan.source(gid)
        assert "fg_jit_" in src
        _compile(src)


def test_random_dag_programs_compile():
    spec = W.random_dag(2, **W.CONFIGS["random_dag"]["small"])
    plan = graph_from_spec(spec).build()
    srcs = sorted({plan.source(g) for g in range(plan.n_groups)}, key=len)
    for s in srcs[-3:] + srcs[:1]:     # the largest programs and one small one
        _compile(s)


def test_tuple_programs_compile():
    """Groups holding a tuple: row selects (the frame's layout) and column
    selects (a transposed concatenation), fields at shifted boxes."""
    for transpose in (False, True):
        g = W.GraphSpec()
        a = g.op("relu", (g.input((40, 32)),))
        b = g.op("exp", (g.input((24, 32)),))
        c = g.op("concat", (g.op("tuple", (a, b)),))
        if transpose:
            c = g.op("transpose", (c,))
        g.mark_output(g.op("scale", (c,), (0.5,)))
        plan = graph_from_spec(g).build()
        assert plan.n_groups == 1
        _compile(plan.source(0))


@pytest.mark.parametrize("shape,kb,tn", [(0, 2, 256), (1 << 16, 2, 256), (2 << 16, 2, 256), (1 << 18, 1, 256),
                                         ((2 << 16) | (1 << 18), 1, 256), (2 << 22, 2, 128),
                                         ((2 << 22) | (1 << 18), 1, 128)])
def test_gemm_cluster_shapes_compile(shape, kb, tn):
    """The GEMM-epilogue program always runs CTA pairs (bits 16-17 of the
    flags are ignored), with one or two K blocks per ring slot and 256- or
    128-column pair tiles; no operand copy is multicast."""
    spec = W.sf_update(256, 256, 512)
    plan = graph_from_spec(spec).build(flags=shape)
    assert plan.groups[0].kind == "gemm"
    src = plan.source(0)
    assert "__cluster_dims__(fg::kGemmCluster, 1, 1)" in src
    assert f"gemm_body<fg::JitEpi, {kb}, {tn}>" in src
    _compile(src)
