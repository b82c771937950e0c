"""The data-parallel exchange around tensor fusion, on CPU with two gloo
ranks (DisCo, Background: gradients from every device are aggregated with an
AllReduce; Introduction: small tensors are fused before it; Related Work:
Horovod's threshold buckets).  Each rank plans its buckets with the library's
host planner and lays the fusion buffer out with the library's host layout
(the byte ranges the device path all-reduces), packs its own gradients into
it with scale 1/N (the oracle's arithmetic: no GPU here) in f32, all-reduces
every bucket's byte range on its own, unpacks, and must hold the exact mean
of both ranks' gradients."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
dist = pytest.importorskip("torch.distributed")

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=WORLD)
        import workloads as W
        from oracle import pack as PK
        from group_execution_gb300 import plan_threshold, layout_offsets

        sizes = [int(x) for x in W.tensor_fusion_sizes(0)[:48]]
        xs = W.tensor_fusion_inputs(sizes, 100 + rank)
        bounds = plan_threshold(sizes, 1 << 20, "f32")
        # every rank must cut the same buckets
        allb = [None] * WORLD
        dist.all_gather_object(allb, bounds)
        assert all(b == bounds for b in allb)
        assert len(bounds) - 1 >= 3

        scale = 1.0 / WORLD
        offs, total = layout_offsets(sizes, "f32")
        # the library's layout is the one the oracle's pack writes
        ref_offs, ref_total = PK.layout(sizes, 4)
        assert list(offs) == list(ref_offs) and total == ref_total
        buf = torch.from_numpy(PK.pack(xs, scale, "f32"))
        assert buf.numel() == total
        starts = [offs[b] if b < len(sizes) else total for b in bounds]
        for k in range(len(bounds) - 1):
            view = buf[starts[k]:starts[k + 1]].view(torch.float32)
            dist.all_reduce(view, op=dist.ReduceOp.SUM)
        got = PK.unpack(buf.numpy(), sizes, 1.0, "f32")

        # the exact mean: both scaled terms, one float32 addition (a sum of
        # two terms does not depend on the order)
        others = [W.tensor_fusion_inputs(sizes, 100 + r) for r in range(WORLD)]
        for i in range(len(sizes)):
            t = [(o[i].astype(np.float64) * scale).astype(np.float32) for o in others]
            ref = (t[0] + t[1]).astype(np.float32)
            np.testing.assert_array_equal(got[i], ref)
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except BaseException as e:  # report, never hang the parent
        q.put((rank, repr(e)))


def test_bucketed_allreduce_two_ranks():
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    ps = [mp.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=240) for _ in range(WORLD))
    for p in ps:
        p.join(timeout=60)
    assert res == {0: "ok", 1: "ok"}, res
