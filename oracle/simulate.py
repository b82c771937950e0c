"""Per-iteration time of a training step with AllReduce communication (test
infrastructure: only tests, the smoke check and the bench's CPU legs use
this module).

DisCo, Simulator: a ready queue holds the computation operators whose
dependencies have cleared; the operator at its head is removed, its
completion time follows from its predecessors' completion times and its own
execution time, and successors whose dependencies have all cleared are
appended at the tail.  AllReduce instructions run in the order their
(possibly fused) gradient tensors are produced; one starts once every tensor
it carries has been produced and the communication channel is free, and it
overlaps with computation.  DisCo, Profiler: an AllReduce of x bytes takes
T = C*x + D (for a ring over N devices with the narrowest link bandwidth B,
C = 2(N-1)/(B*N)).

Readings where the pages are silent: the device runs one computation
operator at a time, in queue order, starting it when the device is free and
its inputs exist; the queue starts with the operators without dependencies in
index order, and successors are appended in index order; a computation
operator may also wait for AllReduces (a parameter update reading the
aggregated gradient): it joins the queue once those AllReduces are
scheduled and starts no earlier than their completion;
AllReduces whose tensors are complete at the same time go in bucket order;
a bucket's bytes are its tensors' bytes added in bucket order and its time
is (start + C*bytes) + D in double precision, one rounding per operation;
the iteration ends when the last operator or AllReduce completes.
"""
from __future__ import annotations

from collections import deque


def ring_coefficient(n_devices, bandwidth):
    """C of T = C*x + D for a ring AllReduce (DisCo, Profiler)."""
    return 2.0 * (n_devices - 1) / (bandwidth * n_devices)


def simulate(op_time, edges, tensor_producer, tensor_bytes, buckets, c, d, ar_edges=()):
    """op_time[i]: execution time of operator i; edges: (src, dst) operator
    dependencies; tensor_producer[t], tensor_bytes[t]: the gradient tensors;
    buckets: list of tensor lists, one fused AllReduce each; ar_edges:
    (bucket, operator) dependencies.  Returns (total, op_finish, ar_start,
    ar_finish)."""
    n = len(op_time)
    preds = [[] for _ in range(n)]
    succ = [[] for _ in range(n)]
    for s, t in edges:
        preds[t].append(s)
        succ[s].append(t)
    ar_wait = [[] for _ in range(n)]
    for b, t in ar_edges:
        ar_wait[t].append(b)
    nb = len(buckets)
    readers = [[] for _ in range(nb)]
    for b, t in ar_edges:
        readers[b].append(t)
    pending = [len(preds[i]) + len(ar_wait[i]) for i in range(n)]
    # tensors still to be produced, per bucket
    left = [len(bk) for bk in buckets]
    bucket_of_producer = [[] for _ in range(n)]
    for b, bk in enumerate(buckets):
        for t in bk:
            bucket_of_producer[tensor_producer[t]].append(b)

    finish = [None] * n
    ar_start, ar_finish = [None] * nb, [None] * nb
    produced_at = [None] * nb
    device = 0.0
    channel = 0.0
    queue = deque(i for i in range(n) if pending[i] == 0)
    complete_buckets = []          # (time, bucket) not yet started

    def run_allreduces(upto):
        """Start, in production order, every AllReduce whose tensors exist."""
        nonlocal channel
        complete_buckets.sort()
        while complete_buckets and complete_buckets[0][0] <= upto:
            t, b = complete_buckets.pop(0)
            ar_start[b] = max(t, channel)
            x = 0.0
            for t_ in buckets[b]:              # the bucket's bytes, added in bucket order
                x += tensor_bytes[t_]
            ar_finish[b] = ar_start[b] + c * x + d
            channel = ar_finish[b]
            for r in sorted(readers[b]):
                pending[r] -= 1
                if pending[r] == 0:
                    queue.append(r)

    for b in range(nb):            # a bucket of no tensors is ready at once
        if left[b] == 0:
            produced_at[b] = 0.0
            complete_buckets.append((0.0, b))
    run_allreduces(0.0)
    done = 0
    while done < n:
        if not queue:
            # the device waits for an AllReduce some operator needs
            if not complete_buckets:
                raise ValueError("dependency cycle or an operator waiting for an AllReduce that never runs")
            run_allreduces(float("inf"))
            continue
        i = queue.popleft()
        ready = max([device] + [finish[p] for p in preds[i]] + [ar_finish[b] for b in ar_wait[i]])
        finish[i] = ready + op_time[i]
        device = finish[i]
        done += 1
        for b in bucket_of_producer[i]:
            left[b] -= 1
            if left[b] == 0:
                produced_at[b] = finish[i]
                complete_buckets.append((finish[i], b))
        for s in sorted(succ[i]):
            pending[s] -= 1
            if pending[s] == 0:
                queue.append(s)
        run_allreduces(device)
    run_allreduces(float("inf"))
    total = max([device] + [f for f in ar_finish if f is not None])
    return total, finish, ar_start, ar_finish
