"""Pins for the oracle's op-by-op executor: per-operator results checked
against IEEE float32 arithmetic, exact integer cases, mathematical identities
and a different construction of the matmul (sum of outer products, the
sufficient-factor form in TAG)."""
import math

import numpy as np

from oracle import execute as E
import workloads as W

rng = np.random.default_rng(1234)


def f32(*shape, lo=-4, hi=4):
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def test_binary_ops_equal_ieee_float32():
    """float64 compute + one rounding == the float32 operation itself."""
    a, b = f32(1000), f32(1000)
    b[::7] = 0.0
    with np.errstate(divide="ignore", invalid="ignore"):
        for op, ref in (("add", a + b), ("sub", a - b), ("mul", a * b), ("div", a / b)):
            got = E.apply_op(op, [a, b], ())
            assert got.dtype == np.float32
            np.testing.assert_array_equal(got, ref)


def test_add3_is_two_rounded_adds():
    """(a + b) + c with b far below a's ulp and c = -a: the first rounding
    decides the result, so one rounding of the exact sum would differ."""
    a = rng.uniform(1, 2, 4096).astype(np.float32)
    b = rng.uniform(0, 2.0 ** -22, 4096).astype(np.float32)
    c = -a
    got = E.apply_op("add", [a, b, c], ())
    np.testing.assert_array_equal(got, (a + b) + c)
    assert not np.array_equal(got, b)


def test_scale_addc_neg_relu():
    x = f32(777)
    np.testing.assert_array_equal(E.apply_op("scale", [x], (0.01,)), np.float32(0.01) * x)
    np.testing.assert_array_equal(E.apply_op("addc", [x], (0.5,)), x + np.float32(0.5))
    np.testing.assert_array_equal(E.apply_op("neg", [x], ()), -x)
    r = E.apply_op("relu", [x], ())
    np.testing.assert_array_equal(r - E.apply_op("relu", [-x], ()), x)
    assert (r >= 0).all()


def test_transcendentals_against_scalar_math():
    x = f32(300, lo=-30, hi=30)
    for op, fn in (("exp", math.exp), ("tanh", math.tanh),
                   ("sigmoid", lambda t: 1.0 / (1.0 + math.exp(-t)))):
        got = E.apply_op(op, [x], ())
        ref = np.array([fn(float(t)) for t in x], dtype=np.float64)
        # correctly rounded float32 of the exact value: within half an ulp
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(got - ref) <= 0.5 * ulp + 1e-300), op


def test_sigmoid_tanh_identity():
    x = f32(1000, lo=-10, hi=10)
    s = E.apply_op("sigmoid", [x], ()).astype(np.float64)
    t = E.apply_op("tanh", [(x / 2).astype(np.float32)], ()).astype(np.float64)
    assert np.max(np.abs(s - (1 + t) / 2)) < 2e-7


def test_broadcasts():
    x = f32(6, 10)
    vc, vr = f32(10), f32(6)
    np.testing.assert_array_equal(E.apply_op("badd_col", [x, np.zeros(10, np.float32)], ()), x)
    np.testing.assert_array_equal(E.apply_op("bmul_col", [x, np.ones(10, np.float32)], ()), x)
    np.testing.assert_array_equal(E.apply_op("badd_col", [x, vc], ())[3], x[3] + vc)
    np.testing.assert_array_equal(
        E.apply_op("badd_row", [x, vr], ()),
        E.apply_op("badd_col", [x.T.copy(), vr], ()).T)
    np.testing.assert_array_equal(E.apply_op("bmul_row", [x, vr], ())[:, 4], x[:, 4] * vr)


def test_injective_round_trips():
    x = f32(6, 10)
    t = E.apply_op("transpose", [x], ())
    assert t.shape == (10, 6) and t[3, 2] == x[2, 3]
    np.testing.assert_array_equal(E.apply_op("transpose", [t], ()), x)
    r = E.apply_op("reshape", [x], (10, 6))
    assert r[1, 0] == x[0, 6]
    np.testing.assert_array_equal(E.apply_op("reshape", [r], (6, 10)), x)


def test_reductions_exact_on_integers():
    x = rng.integers(-1000, 1000, size=(7, 333)).astype(np.float32)
    s = E.apply_op("rowsum", [x], ())
    assert s.tolist() == [float(sum(int(v) for v in row)) for row in x]
    m = E.apply_op("rowmax", [x], ())
    assert m.tolist() == [float(max(row)) for row in x]


def test_rowsum_accumulates_in_float64():
    """1 + 2^-24 * k: float32 accumulation would lose every small term."""
    x = np.full((1, 4097), 2.0 ** -24, dtype=np.float32)
    x[0, 0] = 1.0
    assert E.apply_op("rowsum", [x], ())[0] == np.float32(1.0 + 4096 * 2.0 ** -24)


def test_matmul_equals_sum_of_outer_products():
    """G = U^T V equals the sum over the batch of u_b v_b^T (TAG, sufficient
    factors)."""
    spec = W.sf_update(48, 40, 24)
    u, v = (W.make_input(spec, i) for i in (0, 1))
    g = E.apply_op("matmul_bf16", [u, v], (1, 0))
    acc = np.zeros((40, 24))
    for b in range(48):
        acc += np.outer(u[b].astype(np.float64), v[b].astype(np.float64))
    assert g.shape == (40, 24)
    assert np.max(np.abs(g - acc) / np.maximum(np.abs(acc), 1e-3)) < 1e-6


def test_matmul_exact_on_small_integers():
    a = rng.integers(-8, 8, size=(5, 9)).astype(np.float32)
    b = rng.integers(-8, 8, size=(9, 4)).astype(np.float32)
    ref = [[sum(int(a[i, k]) * int(b[k, j]) for k in range(9)) for j in range(4)] for i in range(5)]
    assert E.apply_op("matmul_bf16", [a, b], (0, 0)).tolist() == ref
    assert E.apply_op("matmul_bf16", [a.T.copy(), b.T.copy()], (1, 1)).tolist() == ref


def test_run_unfused_keeps_outputs_only():
    spec = W.diamond(8, 4)
    ins = W.make_inputs(spec)
    out = E.run_unfused(spec, ins)
    assert list(out) == spec.outputs and out[spec.outputs[0]].shape == (4, 8)
    # transposing the output back gives the pre-transpose sum
    allv = E.run_unfused(spec, ins, keep=[v.vid for v in spec.ops])
    np.testing.assert_array_equal(allv[spec.outputs[0]].T, allv[spec.outputs[0] - 1])
