"""Unfused, op-by-op execution: the semantics fusion must preserve.

Op fusion changes only where intermediate results live, never what is
computed (DisCo, Introduction: fused ops keep intermediates out of device
memory; TVM "Operator Fusion", FuseTIR: the merged function drops the
intermediate buffers).  So the reference result of a fused group is the
result of running its operators one at a time.

Arithmetic: each operator computes in float64 from its float32 (or exact
bfloat16) operands and rounds its result to float32 once.  For +, -, * and /
of two float32 values this equals the IEEE float32 operation (float64 holds
more than twice float32's precision, so the double rounding is harmless).
A three-operand add is two adds, left to right, each rounded.  Reductions
accumulate in float64; the maximum is exact.  The matmul multiplies the exact
bfloat16 values in float64.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def _f(x):
    return np.asarray(x, dtype=np.float64)


def _r(x):
    return np.asarray(x, dtype=np.float64).astype(F32)


def apply_op(op, args, attrs):
    """One operator on float32 operands (float32 result)."""
    a = [_f(x) for x in args]
    if op == "add":
        acc = _r(a[0] + a[1])
        for extra in a[2:]:
            acc = _r(_f(acc) + extra)
        return acc
    if op == "sub":
        return _r(a[0] - a[1])
    if op == "mul":
        return _r(a[0] * a[1])
    if op == "div":
        with np.errstate(divide="ignore", invalid="ignore"):
            return _r(a[0] / a[1])
    if op == "scale":
        return _r(_f(F32(attrs[0])) * a[0])
    if op == "addc":
        return _r(a[0] + _f(F32(attrs[0])))
    if op == "relu":
        return _r(np.where(a[0] > 0, a[0], 0.0))
    if op == "exp":
        with np.errstate(over="ignore"):
            return _r(np.exp(a[0]))
    if op == "sigmoid":
        with np.errstate(over="ignore"):
            return _r(1.0 / (1.0 + np.exp(-a[0])))
    if op == "tanh":
        return _r(np.tanh(a[0]))
    if op == "neg":
        return _r(-a[0])
    if op == "badd_col":
        return _r(a[0] + a[1][None, :])
    if op == "bmul_col":
        return _r(a[0] * a[1][None, :])
    if op == "badd_row":
        return _r(a[0] + a[1][:, None])
    if op == "bmul_row":
        return _r(a[0] * a[1][:, None])
    if op == "tuple":
        return np.ascontiguousarray(np.concatenate([np.asarray(x, dtype=F32) for x in args], axis=0))
    if op == "concat":
        return np.ascontiguousarray(np.asarray(args[0], dtype=F32))
    if op == "transpose":
        return np.ascontiguousarray(args[0].T)
    if op == "reshape":
        return np.ascontiguousarray(args[0].reshape(int(attrs[0]), int(attrs[1])))
    if op == "rowsum":
        return _r(a[0].sum(axis=1))
    if op == "rowmax":
        return args[0].max(axis=1).astype(F32)
    if op == "matmul_bf16":
        A = a[0].T if int(attrs[0]) else a[0]
        B = a[1].T if int(attrs[1]) else a[1]
        return _r(A @ B)
    if op == "opaque_copy":
        return args[0].copy()
    raise ValueError(op)


def run_unfused(spec, inputs, keep=None):
    """Execute every operator in creation order.

    inputs: {vid: float32 array}.  Returns {vid: float32 array} for the
    values in `keep` (default: the graph outputs); other intermediates are
    dropped as soon as their last consumer has run.
    """
    keep = set(spec.outputs if keep is None else keep)
    last_use = {}
    for v in spec.values:
        if not v.is_input:
            for a in v.args:
                last_use[a] = v.vid
    env = {vid: np.asarray(x, dtype=F32) for vid, x in inputs.items()}
    for v in spec.values:
        if v.is_input:
            continue
        env[v.vid] = apply_op(v.op, [env[a] for a in v.args], v.attrs)
        for a in set(v.args):
            if last_use.get(a) == v.vid and a not in keep and not spec.values[a].is_input:
                del env[a]
    return {vid: env[vid] for vid in keep}
