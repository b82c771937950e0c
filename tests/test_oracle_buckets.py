"""Pins for the oracle's AllReduce bucket planning: threshold fusion checked
against an exhaustive search over every contiguous partition (tiny inputs),
closed forms and special cases; neighbour combination against its
definition on boundaries."""
import itertools

import numpy as np
import pytest

from oracle import buckets as B
from oracle import pack as PK
import workloads as W


def _all_partitions(n):
    """Every split of n ordered tensors into non-empty contiguous runs."""
    for cuts in itertools.product((0, 1), repeat=n - 1):
        yield [0] + [i + 1 for i, c in enumerate(cuts) if c] + [n]


def _greedy_valid(sizes, bounds, T):
    """The two properties that characterise greedy threshold fusion: (a) a
    bucket stays within T unless it holds one tensor; (b) no bucket could
    have taken the next bucket's first tensor."""
    tot = [sum(sizes[bounds[k]:bounds[k + 1]]) for k in range(len(bounds) - 1)]
    for k in range(len(tot)):
        if tot[k] > T and bounds[k + 1] - bounds[k] > 1:
            return False
        if k + 1 < len(tot) and tot[k] + sizes[bounds[k + 1]] <= T:
            return False
    return True


@pytest.mark.parametrize("seed", range(40))
def test_threshold_matches_exhaustive_search(seed):
    r = np.random.default_rng(seed)
    n = int(r.integers(1, 10))
    numels = [int(x) for x in r.integers(0, 2000, size=n)]
    T = int(r.choice([0, 256, 512, 1024, 2048, 4096, 10 ** 6]))
    sizes = B.padded_sizes(numels)
    valid = [b for b in _all_partitions(n) if _greedy_valid(sizes, b, T)]
    assert len(valid) == 1, valid          # the properties single out one partition
    assert B.threshold_buckets(numels, T) == valid[0]


def test_threshold_closed_form_equal_sizes():
    # 100 tensors of 1000 bf16 elements span 2048 bytes each: a 10 000-byte
    # threshold holds floor(10000/2048) = 4 per bucket, 25 buckets
    b = B.threshold_buckets([1000] * 100, 10_000)
    assert b == list(range(0, 101, 4))


def test_threshold_special_cases():
    sizes = W.tensor_fusion_sizes(0)
    n = len(sizes)
    assert B.threshold_buckets(sizes, 0) == list(range(n + 1))           # nothing fits: one per tensor
    total = PK.layout(sizes)[1]
    assert B.threshold_buckets(sizes, total) == [0, n]                    # everything fits: one bucket
    assert B.threshold_buckets([10 ** 7, 1, 1], 1024) == [0, 1, 3]        # an oversized tensor sits alone
    assert B.threshold_buckets([], 1024) == [0]


def test_buckets_cover_the_layout():
    sizes = W.tensor_fusion_sizes(0)
    for T in (1 << 20, 8 << 20, 16 << 20):
        b = B.threshold_buckets(sizes, T)
        rng = B.bucket_ranges(sizes, b)
        offs, total = PK.layout(sizes)
        assert rng[0][0] == 0 and rng[-1][1] == total
        assert all(e == s2 for (_, e), (s2, _) in zip(rng, rng[1:]))
        for k, (s, e) in enumerate(rng):
            assert s == offs[b[k]] and s % 256 == 0
            assert e - s <= T or b[k + 1] - b[k] == 1


def test_merge_neighbours():
    b = [0, 3, 5, 9, 12]
    assert B.merge_neighbours(b, 0) == [0, 5, 9, 12]
    assert B.merge_neighbours(b, 2) == [0, 3, 5, 12]
    with pytest.raises(ValueError):
        B.merge_neighbours(b, 3)
    # merging every neighbour pair in turn ends in one bucket
    while len(b) > 2:
        b = B.merge_neighbours(b, 0)
    assert b == [0, 12]
