"""Pins the oracle's composition of operators (its whole-tensor execution in
creation order, with intermediates dropped after their last use) against an
independent evaluator.

The evaluator computes one output element at a time by recursion from the
graph's outputs back to its inputs, from each operator's definition written
as an index map on scalars: an elementwise operator reads its operands at the
same index, a column broadcast reads its vector at the column and a row
broadcast at the row, a transpose swaps the indices, a row-major reshape maps
through the flat index, and a row reduction walks the row.  Each operator's
result is rounded to float32, as the oracle's arithmetic rule states (TVM
"Operator Fusion": fusion changes where intermediates live, not what is
computed; the reference result is the operators run one at a time).  No code
is shared with the oracle: a mistake in its wiring (operand order, the
values a transposed or reshaped operand reads, a value dropped or reused too
early) changes elements that the recursion computes from the graph alone.
"""
import math

import numpy as np
import pytest

import workloads as W
from oracle import execute as OE


def _f32(x):
    return float(np.float32(x))


class _Scalar:
    """Memoised element-by-element evaluation of a graph."""

    def __init__(self, spec, inputs):
        self.spec, self.inputs, self.memo = spec, inputs, {}

    def at(self, vid, idx):
        key = (vid, idx)
        if key not in self.memo:
            v = self.spec.values[vid]
            self.memo[key] = float(self.inputs[vid][idx]) if v.is_input else self._op(v, idx)
        return self.memo[key]

    def _op(self, v, idx):
        op, a = v.op, v.args
        src = self.spec.values[a[0]]
        if op == "add":
            acc = _f32(self.at(a[0], idx) + self.at(a[1], idx))
            for extra in a[2:]:
                acc = _f32(acc + self.at(extra, idx))
            return acc
        if op == "sub":
            return _f32(self.at(a[0], idx) - self.at(a[1], idx))
        if op == "mul":
            return _f32(self.at(a[0], idx) * self.at(a[1], idx))
        if op == "scale":
            return _f32(_f32(v.attrs[0]) * self.at(a[0], idx))
        if op == "addc":
            return _f32(self.at(a[0], idx) + _f32(v.attrs[0]))
        if op == "neg":
            return -self.at(a[0], idx)
        if op == "relu":
            x = self.at(a[0], idx)
            return x if x > 0 else 0.0
        if op == "exp":
            return _f32(math.exp(self.at(a[0], idx)))
        if op == "sigmoid":
            x = self.at(a[0], idx)
            return 0.0 if -x > 700.0 else _f32(1.0 / (1.0 + math.exp(-x)))
        if op == "tanh":
            return _f32(math.tanh(self.at(a[0], idx)))
        if op in ("badd_col", "bmul_col", "badd_row", "bmul_row"):
            i, j = idx
            b = self.at(a[1], (j,) if op.endswith("col") else (i,))
            x = self.at(a[0], idx)
            return _f32(x + b if op.startswith("badd") else x * b)
        if op == "transpose":
            i, j = idx
            return self.at(a[0], (j, i))
        if op == "reshape":
            i, j = idx
            flat = i * v.shape[1] + j
            return self.at(a[0], (flat // src.shape[1], flat % src.shape[1]))
        if op == "rowsum":
            (i,) = idx
            return _f32(math.fsum(self.at(a[0], (i, j)) for j in range(src.shape[1])))
        if op == "rowmax":
            (i,) = idx
            return max(self.at(a[0], (i, j)) for j in range(src.shape[1]))
        raise ValueError(op)


def _compare(spec, seed):
    inputs = W.make_inputs(spec, seed)
    ref = OE.run_unfused(spec, inputs)
    ev = _Scalar(spec, inputs)
    n = 0
    for vid in spec.outputs:
        got = ref[vid]
        want = np.array([ev.at(vid, idx) for idx in np.ndindex(*got.shape)], dtype=np.float64).reshape(got.shape)
        # both sides round every operator's result to float32; they may part
        # only where a transcendental or a float64 sum lands within a float64
        # rounding of a float32 boundary
        scale = np.maximum(1.0, np.abs(want))
        bad = np.abs(got.astype(np.float64) - want) > 4e-7 * scale
        assert not bad.any(), (vid, spec.values[vid].op, np.argwhere(bad)[:5])
        n += got.size
    return n


@pytest.mark.parametrize("seed", range(4))
def test_random_dag_composition(seed):
    """Random DAGs with every operator kind of the generator (elementwise of
    arity 1-3, column broadcasts, transposes, reshapes between [R,C] and
    [C,R], row sums and maxima), scaled down with the full-size graph."""
    spec = W.random_dag(seed, n_ops=120, R=12, C=8, nominal_R=8192, nominal_C=4096)
    ops = {v.op for v in spec.ops}
    assert {"transpose", "reshape"} & ops and {"rowsum", "rowmax"} & ops
    assert _compare(spec, seed) > 0


def test_every_operator_composed():
    """A hand-built graph that chains every remaining operator through
    transposes and reshapes, so that each one reads a permuted operand."""
    g = W.GraphSpec()
    x = g.input((6, 4))
    y = g.input((4, 6))
    c = g.input((4,))
    r = g.input((6,))
    t = g.op("transpose", (y,))                       # [6,4]
    d = g.op("sub", (x, t))
    e = g.op("bmul_row", (g.op("badd_row", (d, r)), r))
    f = g.op("scale", (g.op("addc", (g.op("neg", (e,)),), (0.25,)),), (1.5,))
    h = g.op("reshape", (f,), (4, 6))
    k = g.op("add", (h, y, g.op("transpose", (x,))))  # three operands
    m = g.op("bmul_col", (g.op("badd_col", (g.op("reshape", (k,), (6, 4)), c)), c))
    s = g.op("rowsum", (g.op("tanh", (m,)),))
    g.mark_output(g.op("sigmoid", (g.op("mul", (s, r)),)))
    g.mark_output(g.op("rowmax", (g.op("exp", (g.op("transpose", (m,)),)),)))
    g.mark_output(k)
    assert _compare(g, 3) == 6 + 4 + 24
