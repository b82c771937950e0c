"""Helpers for GPU tests: run a plan group by group (fused) or node by node
(unfused) through the C ABI on device tensors."""
from __future__ import annotations

import numpy as np
import torch

from group_execution_gb300 import graph_from_spec


def to_dev(spec, vid, arr):
    t = torch.from_numpy(np.ascontiguousarray(arr)).cuda()
    if spec.values[vid].dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t


def empty_for(spec, vid):
    return torch.empty(spec.values[vid].shape, dtype=torch.float32, device="cuda")


def run_fused(plan, spec, dev_inputs, keep_all=True):
    """Launch every group in order; returns {vid: tensor} of group outputs."""
    env = dict(dev_inputs)
    for gid, info in enumerate(plan.groups):
        for o in info.outs:                  # the sink output and any extra outputs
            env[o] = empty_for(spec, o)
        plan.launch_group(gid, {v: env[v] for v in info.leaves + info.outs})
    return env


def run_unfused(plan, spec, dev_inputs):
    env = dict(dev_inputs)
    node = 0
    for v in spec.values:
        if v.is_input:
            continue
        env[v.vid] = empty_for(spec, v.vid)
        plan.launch_unfused(node, {a: env[a] for a in v.args} | {v.vid: env[v.vid]})
        node += 1
    return env


def prepare(spec, seed=0, flags=None, **build_kw):
    if flags is not None:
        build_kw["flags"] = flags
    import workloads as W
    inputs = W.make_inputs(spec, seed)
    g = graph_from_spec(spec)
    plan = g.build(**build_kw)
    dev = {vid: to_dev(spec, vid, a) for vid, a in inputs.items()}
    return g, plan, inputs, dev
