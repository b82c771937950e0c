"""Pins for the oracle's tensor-fusion layout and bf16 rounding (DisCo,
Introduction: the fused tensor's size is the sum of its parts)."""
import numpy as np
import pytest

from oracle import pack as PK
from tests._helpers import read_golden
import workloads as W


def test_layout_golden():
    d = {ln.split()[0]: [int(x) for x in ln.split()[1].split(",")]
         for ln in read_golden("pack_layout_small.txt")}
    offs, total = PK.layout(d["numels"])
    assert offs == d["offsets"] and total == d["total"][0]


def test_layout_size_is_sum_plus_padding():
    sizes = W.tensor_fusion_sizes(0)
    offs, total = PK.layout(sizes)
    data = int(sizes.sum()) * 2
    assert total >= data and total - data < 256 * len(sizes)
    assert all(o % 256 == 0 for o in offs)
    ends = [o + int(n) * 2 for o, n in zip(offs, sizes)]
    assert all(e <= o2 for e, o2 in zip(ends, offs[1:] + [total]))


def test_bf16_rne_golden():
    for ln in read_golden("bf16_rne.txt"):
        f, b = ln.split()[:2]
        x = np.array([int(f, 16)], dtype=np.uint32).view(np.float32)
        assert PK.bf16_rne_bits(x)[0] == int(b, 16), ln


def test_bf16_rne_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    y = PK.bf16_bits_to_f32(PK.bf16_rne_bits(x))
    assert np.isnan(y).all()


def test_bf16_rne_matches_torch():
    """A library routine with the same definition (torch's float -> bfloat16
    conversion rounds to nearest even)."""
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(5)
    bits = r.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    x = np.concatenate([x, r.normal(0, 1e-3, 1 << 16).astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(PK.bf16_rne_bits(x), ref)


def _tensors(sizes, seed=0):
    return W.tensor_fusion_inputs(sizes, seed)


def test_unpack_pack_is_rounded_scaled_input():
    sizes = [1, 3, 4, 5, 127, 128, 129, 1000]
    xs = _tensors(sizes)
    buf = PK.pack(xs, 0.125)
    ys = PK.unpack(buf, sizes, 1.0)
    for x, y in zip(xs, ys):
        ref = PK.bf16_bits_to_f32(PK.bf16_rne_bits(x * np.float32(0.125)))
        np.testing.assert_array_equal(y, ref)


def test_pack_unpack_is_identity_on_buffer():
    sizes = [1, 3, 4, 5, 127, 128, 129, 1000]
    buf = PK.pack(_tensors(sizes), 0.125)
    again = PK.pack(PK.unpack(buf, sizes, 1.0), 1.0)
    np.testing.assert_array_equal(again, buf)
    offs, total = PK.layout(sizes)
    mask = np.zeros(total, bool)
    for o, n in zip(offs, sizes):
        mask[o:o + 2 * n] = True
    assert (buf[~mask] == 0).all()


def test_fp32_buffer_scale_one_is_identity():
    sizes = [7, 64, 1000]
    xs = _tensors(sizes)
    buf = PK.pack(xs, 1.0, "f32")
    for x, y in zip(xs, PK.unpack(buf, sizes, 1.0, "f32")):
        np.testing.assert_array_equal(x, y)


def test_tensor_fusion_sizes_spec():
    s = W.tensor_fusion_sizes(0)
    assert len(s) == 161 and s.sum() == 25_600_000
    assert s.min() >= 256 and s.max() <= 2_400_000
    assert (s * 4 < (1 << 20)).mean() > 0.5      # "over 50%" small tensors
