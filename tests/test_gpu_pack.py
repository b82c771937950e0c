"""GPU parity of tensor-fusion pack/unpack against the oracle: bit-exact
buffer bytes (data and zero padding) and bit-exact unpacked tensors."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import pack as PK
from group_execution_gb300 import TensorFusion

pytestmark = pytest.mark.gpu


def _run(sizes, scale=0.125, uscale=1.0, buf_dtype="bf16", seed=0):
    xs = W.tensor_fusion_inputs(sizes, seed)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev, buf_dtype)
    offs, total = PK.layout(sizes, 2 if buf_dtype == "bf16" else 4)
    assert tf.offsets == offs and tf.total_bytes == total
    buf = torch.full((total,), 0xAB, dtype=torch.uint8, device="cuda")   # poison padding
    tf.pack(scale, buf)
    torch.cuda.synchronize()
    ref = PK.pack(xs, scale, buf_dtype)
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)
    for d in dev:
        d.fill_(float("nan"))
    tf.unpack(uscale, buf)
    tf.sync()
    back = PK.unpack(ref, sizes, uscale, buf_dtype)
    for d, r in zip(dev, back):
        np.testing.assert_array_equal(d.cpu().numpy(), r)
    return tf


def test_pack_small_ragged():
    _run([1, 3, 4, 5, 127, 128, 129, 1000, 4095, 4096, 4097, 8192 + 7])


def test_pack_empty_tensors():
    _run([5, 0, 8192, 0, 3, 8192 * 2 + 1])
    _run([0, 9, 0], buf_dtype="f32")


def test_pack_config_full():
    _run(W.tensor_fusion_sizes(0))


def test_unpack_scaled_both_buffers():
    # whole chunks (bulk-copied) and partial ones (through registers), with a
    # non-trivial unscale, for both buffer types
    sizes = [8192 * 5, 8192 * 2 + 3, 17, 8192 * 40 + 8]
    _run(sizes, scale=0.25, uscale=0.375, buf_dtype="bf16", seed=5)
    _run(sizes, scale=0.25, uscale=0.375, buf_dtype="f32", seed=6)


def test_pack_fp32_buffer_identity():
    sizes = [7, 64, 5000, 4096 * 3]
    xs = W.tensor_fusion_inputs(sizes, 3)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev, "f32")
    buf = torch.zeros((tf.total_bytes,), dtype=torch.uint8, device="cuda")
    tf.pack(1.0, buf)
    for d in dev:
        d.zero_()
    tf.unpack(1.0, buf)
    tf.sync()
    for d, x in zip(dev, xs):
        np.testing.assert_array_equal(d.cpu().numpy(), x)


def test_pack_special_values():
    x = np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, 1e-45, -1e-40, 1.0 + 2 ** -8, 65504.0], np.float32)
    dev = [torch.from_numpy(x).cuda()]
    tf = TensorFusion(dev)
    buf = torch.zeros((tf.total_bytes,), dtype=torch.uint8, device="cuda")
    tf.pack(1.0, buf)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(buf.cpu().numpy(), PK.pack([x], 1.0))


def test_bucketed_pack_unpack_ranges():
    """Threshold buckets packed and unpacked one launch per bucket: each launch
    writes exactly its bucket's bytes (bit-exact against the oracle) and
    leaves every other byte and tensor alone."""
    from oracle import buckets as OB
    from group_execution_gb300 import plan_threshold
    sizes = W.tensor_fusion_sizes(0)
    xs = W.tensor_fusion_inputs(sizes, 1)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev)
    bounds = plan_threshold(list(sizes), 8 << 20)
    assert bounds == OB.threshold_buckets(list(sizes), 8 << 20)
    nb = len(bounds) - 1
    assert nb >= 4
    rng = tf.bucket_ranges(bounds)
    assert rng == OB.bucket_ranges(list(sizes), bounds)
    ref = PK.pack(xs, 0.125)
    buf = torch.full((tf.total_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
    for k in reversed(range(nb)):                      # last bucket first
        tf.pack_range(bounds[k], bounds[k + 1] - bounds[k], 0.125, buf)
        torch.cuda.synchronize()
        got = buf.cpu().numpy()
        s, e = rng[k]
        np.testing.assert_array_equal(got[s:e], ref[s:e])
        assert (got[:s] == 0xAB).all()                 # earlier buckets untouched so far
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)
    back = PK.unpack(ref, sizes, 2.0, "bf16")
    for d in dev:
        d.fill_(float("nan"))
    for k in range(nb):
        tf.unpack_range(bounds[k], bounds[k + 1] - bounds[k], 2.0, buf)
        tf.sync()
        for i in range(bounds[k], bounds[k + 1]):
            np.testing.assert_array_equal(dev[i].cpu().numpy(), back[i])
        if bounds[k + 1] < len(dev):
            assert torch.isnan(dev[bounds[k + 1]]).all()   # the next bucket is not written yet


def test_range_edge_cases():
    from group_execution_gb300 import FgError
    sizes = [5, 8192 * 2 + 3, 17]
    xs = W.tensor_fusion_inputs(sizes, 2)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev)
    buf = torch.full((tf.total_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
    tf.pack_range(1, 0, 1.0, buf)                      # an empty range launches nothing
    torch.cuda.synchronize()
    assert (buf.cpu().numpy() == 0xAB).all()
    with pytest.raises(FgError):
        tf.pack_range(2, 2, 1.0, buf)
    with pytest.raises(FgError):
        tf.unpack_range(-1, 1, 1.0, buf)
    tf.pack_range(1, 1, 1.0, buf)                      # the middle tensor, padding included
    torch.cuda.synchronize()
    ref = PK.pack(xs, 1.0)
    s, e = tf.offsets[1], tf.offsets[2]
    got = buf.cpu().numpy()
    np.testing.assert_array_equal(got[s:e], ref[s:e])
    assert (got[:s] == 0xAB).all() and (got[e:] == 0xAB).all()


def _bucketed(sizes, threshold, seed=0):
    from group_execution_gb300 import plan_threshold
    xs = W.tensor_fusion_inputs(sizes, seed)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev)
    bounds = plan_threshold(sizes, threshold)
    tf.set_buckets(bounds)
    return tf, bounds, PK.pack(xs, 0.125)


def test_pack_buckets_one_launch():
    """Every AllReduce bucket packed in one launch: the buffer equals the
    oracle's bytes, and after each of three launches every bucket reads as
    ready (its count reached that launch's total each time)."""
    sizes = W.tensor_fusion_sizes(0)
    tf, bounds, ref = _bucketed(sizes, 8 << 20)
    nb = len(bounds) - 1
    assert nb > 3
    for _ in range(3):
        buf = torch.full((tf.total_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
        tf.pack_buckets(0.125, buf)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(buf.cpu().numpy(), ref)
        assert all(tf.bucket_ready(b) for b in range(nb))


def test_pack_buckets_small_and_single():
    """Buckets of one tensor each (empty and ragged tensors included), and a
    single bucket of everything."""
    sizes = [5, 0, 8192, 0, 3, 8192 * 2 + 1, 1]
    for threshold in (0, 1 << 30):
        tf, bounds, ref = _bucketed(sizes, threshold, seed=2)
        assert len(bounds) - 1 == (len(sizes) if threshold == 0 else 1)
        buf = torch.full((tf.total_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
        tf.pack_buckets(0.125, buf)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(buf.cpu().numpy(), ref)
        assert all(tf.bucket_ready(b) for b in range(len(bounds) - 1))


def test_bucket_wait_orders_each_bucket():
    """A second stream waits for each bucket in turn (a stream-ordered wait
    on its count) and copies that bucket's bytes out while the one pack
    launch may still be running: every copy equals the oracle's bytes."""
    sizes = W.tensor_fusion_sizes(0)
    tf, bounds, ref = _bucketed(sizes, 8 << 20)
    ranges = tf.bucket_ranges(bounds)
    s2 = torch.cuda.Stream()
    for _ in range(2):
        buf = torch.full((tf.total_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        tf.pack_buckets(0.125, buf)
        outs = []
        for b, (lo, hi) in enumerate(ranges):
            tf.bucket_wait(b, s2)
            with torch.cuda.stream(s2):
                outs.append(buf[lo:hi].clone())
        torch.cuda.synchronize()
        for (lo, hi), o in zip(ranges, outs):
            np.testing.assert_array_equal(o.cpu().numpy(), ref[lo:hi])


def test_bucket_ready_words_seen_by_a_device_consumer_during_the_launch():
    """A device-side consumer of the bucket counts (one CTA of the pack
    launch, polling each bucket's count in order) sees the first buckets ready while
    other CTAs are still packing: the first bucket well before the launch's
    last packing CTA finishes.  The buffer still holds tf_pack's bytes."""
    from group_execution_gb300 import plan_threshold
    sizes = W.tensor_fusion_sizes(0)
    xs = W.tensor_fusion_inputs(sizes)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev)
    bounds = plan_threshold(list(sizes), 8 << 20)
    nb = len(bounds) - 1
    tf.set_buckets(bounds)
    buf = torch.empty((tf.total_bytes,), dtype=torch.uint8, device="cuda")
    times = torch.zeros(nb + 1, dtype=torch.int64, device="cuda")
    expect = PK.pack(xs, 0.125)
    for _ in range(3):
        times.zero_()
        tf.pack_buckets_observed(0.125, buf, times)
        tf.sync()
        t = times.cpu().numpy()
        assert (t[:nb] > 0).all(), t
        end = t[nb]
        # the first bucket (8 MiB of a 51 MB buffer) is seen ready at least
        # 5 us before the last packing CTA is done
        assert end - t[0] >= 5000, (t - t[0]).tolist()
        assert np.array_equal(buf.cpu().numpy(), expect)


def test_device_consumer_wait_is_bounded_and_reported():
    """Watching for a launch that never comes: every wait of the consumer
    expires after 1 ms, FG_ETIMEOUT is reported once, and the layout then
    packs and reports normally."""
    from group_execution_gb300 import FgError, _lib
    sizes = [5000, 100000, 3000, 70000]
    xs = W.tensor_fusion_inputs(sizes)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev)
    tf.set_buckets([0, 2, 4])
    buf = torch.empty((tf.total_bytes,), dtype=torch.uint8, device="cuda")
    times = torch.zeros(3, dtype=torch.int64, device="cuda")
    tf.pack_buckets_observed(1.0, buf, times, seq_offset=1, wait_limit_ns=1_000_000)
    with pytest.raises(FgError) as e:
        tf.sync()
    assert e.value.status == _lib.FG_ETIMEOUT
    assert times.cpu().numpy()[:2].tolist() == [0, 0]
    tf.sync()                                   # the word was cleared
    tf.pack_buckets_observed(1.0, buf, times)
    tf.sync()
    assert (times.cpu().numpy()[:2] > 0).all()
    assert np.array_equal(buf.cpu().numpy(), PK.pack(xs, 1.0))


def test_pack_of_unpack_reproduces_the_buffer():
    """Unpack then pack with scale 1 gives back the bf16 buffer byte for byte
    (data bytes: bf16 -> fp32 -> bf16 is exact; padding: zero), over ragged
    tensors; with an fp32 buffer, pack then unpack with scale 1 is the
    identity on the tensors."""
    sizes = [1, 7, 8192, 8193, 3 * 8192 - 5, 0, 65536 + 17]
    xs = W.tensor_fusion_inputs(sizes, 4)
    dev = [torch.from_numpy(x).cuda() for x in xs]
    tf = TensorFusion(dev)
    buf = torch.empty((tf.total_bytes,), dtype=torch.uint8, device="cuda")
    tf.pack(0.125, buf)
    tf.unpack(1.0, buf)
    buf2 = torch.full((tf.total_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
    tf.pack(1.0, buf2)
    tf.sync()
    np.testing.assert_array_equal(buf2.cpu().numpy(), buf.cpu().numpy())
    dev32 = [torch.from_numpy(x).cuda() for x in xs]
    tf32 = TensorFusion(dev32, "f32")
    b32 = torch.empty((tf32.total_bytes,), dtype=torch.uint8, device="cuda")
    tf32.pack(1.0, b32)
    for d in dev32:
        d.fill_(float("nan"))
    tf32.unpack(1.0, b32)
    tf32.sync()
    for d, x in zip(dev32, xs):
        np.testing.assert_array_equal(d.cpu().numpy(), x)


def test_bucket_counts_over_many_launches_and_a_new_table():
    """The bucket counts are never reset: after each of 12 bucketed launches
    every bucket reads complete, a stream waiting on the last launch's
    totals passes, and a new bucket table starts the counting over (its
    buckets read complete after its first launch)."""
    from group_execution_gb300 import plan_threshold
    sizes = W.tensor_fusion_sizes(0)[:60]
    tf, bounds, ref = _bucketed(sizes, 2 << 20)
    nb = len(bounds) - 1
    buf = torch.empty((tf.total_bytes,), dtype=torch.uint8, device="cuda")
    s2 = torch.cuda.Stream()
    for _ in range(12):
        tf.pack_buckets(0.125, buf)
        torch.cuda.synchronize()
        assert all(tf.bucket_ready(b) for b in range(nb))
    for b in range(nb):
        tf.bucket_wait(b, s2)
    s2.synchronize()
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)
    bounds2 = plan_threshold(list(sizes), 8 << 20)
    tf.set_buckets(bounds2)
    tf.pack_buckets(0.125, buf)
    torch.cuda.synchronize()
    assert all(tf.bucket_ready(b) for b in range(len(bounds2) - 1))
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)
