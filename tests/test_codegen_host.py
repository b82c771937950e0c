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
