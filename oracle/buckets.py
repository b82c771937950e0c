"""AllReduce buckets over a tensor-fusion layout (test infrastructure: only
tests, the smoke check and the bench's CPU baseline use this module).

Two ways of cutting the gradient list into fused AllReduce tensors:

* Threshold fusion (DisCo, Related Work, on Horovod: small AllReduce tensors
  are combined up to a pre-defined fusion threshold, as XLA's AllReduce
  combiner does; DisCo, Background, on JAX/XLA: AllReduce instructions are
  combined according to a pre-defined tensor size threshold).
* Neighbour combination (DisCo, Strategy Maker, optimisation method (iii):
  an AllReduce instruction is combined with a neighbouring one, neighbours
  being the gradient tensors of adjacent gradient computations).

Readings where the pages are silent: the gradient tensors are given in the
order they are produced, so neighbours are adjacent indices and every bucket
is a contiguous run of tensors; a bucket's size is the number of fusion
buffer bytes it spans (each tensor's bytes rounded up to the layout's
alignment, which is what the fused AllReduce transmits); threshold fusion is
greedy in production order: a tensor joins the open bucket when the bucket
stays within the threshold, otherwise it opens a new one, so a tensor larger
than the threshold sits alone.  Buckets are described by their boundaries:
bucket b holds tensors bounds[b] .. bounds[b+1]-1.
"""
from __future__ import annotations

from oracle.pack import align_up, layout


def padded_sizes(numels, elem_bytes=2, align=256):
    """Bytes each tensor spans in the fusion buffer."""
    return [align_up(int(n) * elem_bytes, align) for n in numels]


def threshold_buckets(numels, threshold, elem_bytes=2, align=256):
    """Greedy threshold fusion in production order; returns the boundaries
    (no tensors: no buckets)."""
    if len(numels) == 0:
        return [0]
    bounds, cur = [0], 0
    for i, s in enumerate(padded_sizes(numels, elem_bytes, align)):
        if i > bounds[-1] and cur + s > threshold:
            bounds.append(i)
            cur = 0
        cur += s
    bounds.append(len(numels))
    return bounds


def merge_neighbours(bounds, j):
    """Bucket j combined with its successor j+1 (one application of the
    neighbour-combination move)."""
    if not 0 <= j < len(bounds) - 2:
        raise ValueError("bucket has no successor")
    return bounds[:j + 1] + bounds[j + 2:]


def bucket_ranges(numels, bounds, elem_bytes=2, align=256):
    """Byte range [start, end) of every bucket in the fusion buffer."""
    offs, total = layout(numels, elem_bytes, align)
    starts = [offs[b] if b < len(numels) else total for b in bounds]
    return [(starts[k], starts[k + 1]) for k in range(len(bounds) - 1)]
