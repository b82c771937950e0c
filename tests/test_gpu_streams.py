"""Streams: launches of one plan are ordered (one stream, or streams ordered
by events); concurrency comes from one plan per stream, since each group owns
device state that a launch uses from its start to its end (tile claim
counter, split partials, arrival counters, split workspace).  Two plans of the
same graph launched at once on two streams must each match the oracle; one
plan whose launches alternate between two streams ordered by events must too.
Replacing a bucket table does not synchronize the device: a pack enqueued
before the replacement and one enqueued after it both give tf_pack's bytes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import execute as OE
from oracle import pack as PK
from tests._helpers import check_parity
from tests._gpu import to_dev, empty_for
from group_execution_gb300 import graph_from_spec, TensorFusion, plan_threshold

pytestmark = pytest.mark.gpu

SPECS = {
    "diamond": lambda: W.diamond(1024, 512),
    "rowsum": lambda: W.rnnlm_chain(4096, 1024),
    "sf_update": lambda: W.sf_update(256, 512, 512),
}


def _env(spec, seed):
    ins = W.make_inputs(spec, seed)
    env = {vid: to_dev(spec, vid, a) for vid, a in ins.items()}
    for v in spec.ops:
        env[v.vid] = empty_for(spec, v.vid)
    return ins, env


def _launch_all(plan, env, stream):
    for gid, gi in enumerate(plan.groups):
        plan.launch_group(gid, {v: env[v] for v in gi.leaves + gi.outs}, stream=stream)


def _check(spec, ins, env):
    ref = OE.run_unfused(spec, ins)
    for o in spec.outputs:
        check_parity(spec, o, env[o].cpu().numpy(), ref[o])


@pytest.mark.parametrize("name", list(SPECS))
def test_two_plans_concurrently_on_two_streams(name):
    spec = SPECS[name]()
    g = graph_from_spec(spec)
    plans = [g.build(), g.build()]
    data = [_env(spec, seed) for seed in (1, 2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(5):
        for p, (ins, env), st in zip(plans, data, streams):
            _launch_all(p, env, st)
    torch.cuda.synchronize()
    for p, st in zip(plans, streams):
        p.sync(st)
    for ins, env in data:
        _check(spec, ins, env)


@pytest.mark.parametrize("name", list(SPECS))
def test_one_plan_on_two_streams_ordered_by_events(name):
    spec = SPECS[name]()
    plan = graph_from_spec(spec).build()
    data = [_env(spec, seed) for seed in (3, 4)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    prev = None
    for k in range(6):
        st = streams[k % 2]
        if prev is not None:
            st.wait_event(prev)
        _launch_all(plan, data[k % 2][1], st)
        prev = torch.cuda.Event()
        prev.record(st)
    torch.cuda.synchronize()
    plan.sync()
    for ins, env in data:
        _check(spec, ins, env)


def test_bucket_table_replaced_without_synchronizing():
    sizes = W.tensor_fusion_sizes(0)[:40]
    xs = W.tensor_fusion_inputs(sizes)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev)
    expect = PK.pack(xs, 0.125)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    bufs = [torch.empty((tf.total_bytes,), dtype=torch.uint8, device="cuda") for _ in range(3)]
    torch.cuda.synchronize()
    for thr, buf in zip((1 << 20, 4 << 20, 1 << 22), bufs):
        tf.set_buckets(plan_threshold(list(sizes), thr))
        tf.pack_buckets(0.125, buf, stream=s1)
        tf.bucket_wait(0, stream=s2)      # a stream wait that reads the table
    torch.cuda.synchronize()
    for buf in bufs:
        assert np.array_equal(buf.cpu().numpy(), expect)
