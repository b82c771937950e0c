"""Pins for the oracle's training-step simulator (DisCo, Simulator and
Profiler): hand-worked schedules, the ring AllReduce formula, and the rules
of the schedule checked on random instances."""
import math

import numpy as np
import pytest

from oracle import simulate as OS


def test_chain_one_bucket_per_tensor():
    # ops 1, 2, 3 in a chain, each producing one tensor of 10, 20, 30 bytes;
    # T = 0.1 x + 0.5: AR0 1 -> 2.5, AR1 3 -> 5.5, AR2 6 -> 9.5
    tot, fin, s, f = OS.simulate([1, 2, 3], [(0, 1), (1, 2)], [0, 1, 2], [10, 20, 30],
                                 [[0], [1], [2]], 0.1, 0.5)
    assert fin == [1, 3, 6]
    assert s == [1, 3, 6] and f == pytest.approx([2.5, 5.5, 9.5])
    assert tot == pytest.approx(9.5)


def test_fused_tensor_waits_for_all_parts():
    tot, _, s, f = OS.simulate([1, 2, 3], [(0, 1), (1, 2)], [0, 1, 2], [10, 20, 30],
                               [[0, 1, 2]], 0.1, 0.5)
    assert s == [6] and f == pytest.approx([12.5]) and tot == pytest.approx(12.5)


def test_channel_is_used_in_production_order():
    # one op produces two tensors: the second AllReduce waits for the channel
    tot, _, s, f = OS.simulate([1], [], [0, 0], [10, 10], [[0], [1]], 0.1, 0.5)
    assert s == pytest.approx([1, 2.5]) and f == pytest.approx([2.5, 4.0])


def test_fifo_ready_queue_and_overlap():
    # op0 -> {op1, op2} -> op3; FIFO runs op1 before op2; op2's tensor is
    # reduced while op3 computes
    tot, fin, s, f = OS.simulate([1, 5, 1, 1], [(0, 1), (0, 2), (1, 3), (2, 3)], [2], [10], [[0]], 0.1, 0.0)
    assert fin == [1, 6, 7, 8] and s == [7] and f == pytest.approx([8.0])
    assert tot == pytest.approx(8.0)


def test_update_waits_for_its_allreduce():
    # op1 (the update) reads bucket 0's result: it starts when the AllReduce ends
    tot, fin, s, f = OS.simulate([2, 1], [], [0], [100], [[0]], 0.1, 1.0, ar_edges=[(0, 1)])
    assert f == pytest.approx([13.0]) and fin == pytest.approx([2, 14]) and tot == pytest.approx(14)


def test_ring_coefficient():
    # each rank sends and receives 2(N-1)/N of the tensor over its slowest link
    c = OS.ring_coefficient(8, 100.0)
    assert c == pytest.approx(2 * 7 / 800)
    assert OS.ring_coefficient(1, 5.0) == 0.0


@pytest.mark.parametrize("seed", range(40))
def test_schedule_rules_on_random_instances(seed):
    r = np.random.default_rng(seed)
    n = int(r.integers(1, 25))
    edges = sorted({(int(a), int(b)) for a, b in r.integers(0, n, size=(2 * n, 2)) if a < b})
    times = r.uniform(0.1, 3.0, size=n).tolist()
    nt = int(r.integers(0, 12))
    prod = r.integers(0, n, size=nt).tolist()
    by = r.uniform(1, 100, size=nt).tolist()
    order = r.permutation(nt).tolist()
    cuts = sorted(set(r.integers(0, nt + 1, size=3).tolist()) | {0, nt})
    buckets = [order[a:b] for a, b in zip(cuts, cuts[1:]) if b > a]
    ar_edges = [(int(b), int(t)) for b, t in zip(r.integers(0, max(1, len(buckets)), size=2),
                                                   r.integers(0, n, size=2))
                if len(buckets) and all(prod[x] < t for x in buckets[int(b)])]
    c, d = 0.01, 0.2
    tot, fin, s, f = OS.simulate(times, edges, prod, by, buckets, c, d, ar_edges)
    start = [fin[i] - times[i] for i in range(n)]
    for a, b in edges:
        assert start[b] >= fin[a] - 1e-12
    for b, t in ar_edges:
        assert start[t] >= f[b] - 1e-12
    seq = sorted(range(n), key=lambda i: start[i])
    for a, b in zip(seq, seq[1:]):
        assert start[b] >= fin[a] - 1e-12                    # one operator at a time
    produced = [max(fin[prod[x]] for x in bk) for bk in buckets]
    for b, bk in enumerate(buckets):
        assert s[b] >= produced[b] - 1e-12
        assert f[b] == pytest.approx(s[b] + c * sum(by[x] for x in bk) + d)
    ar_seq = sorted(range(len(buckets)), key=lambda b: s[b])
    for a, b in zip(ar_seq, ar_seq[1:]):
        assert s[b] >= f[a] - 1e-12                          # one AllReduce at a time
        assert produced[b] >= produced[a] - 1e-12            # in production order
    for b in range(len(buckets)):                            # no needless channel idling
        prev = max([f[a] for a in range(len(buckets)) if s[a] < s[b]], default=0.0)
        assert s[b] == pytest.approx(max(produced[b], prev))
    assert tot == pytest.approx(max(fin + f + [0.0]))
