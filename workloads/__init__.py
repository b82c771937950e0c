"""Seeded synthetic workloads: graph descriptions and their input tensors.

This module is shared by the CPU oracle and by the GPU path, and therefore holds
none of the method's arithmetic: no operator semantics, no pattern kinds, no
post-dominator or grouping logic, no rounding.  It only says *which* graph to
build (operator names, operands, attributes, shapes) and draws the input
values from seeded NumPy generators.

Shapes follow the workloads the pages describe: the RNNLM Mul1/Mul2/Sigmoid
chain (DisCo, Introduction, Fig. 2), the diamond a post-dominator pass must
close (TVM "Operator Fusion", FuseOps > Algorithm), a matmul with an
elementwise tail (TVM, Fusion rules, phase 0) instantiated as the
sufficient-factor gradient G = U^T V of TAG (Sec. on sufficient factor
broadcasting), the many-small-tensor gradient set of tensor fusion (DisCo,
Introduction), and a seeded random DAG.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# Operator vocabulary (names only; semantics live in the oracle and in the
# CUDA library, each written separately).
OPS = (
    "add", "sub", "mul", "div", "scale", "addc", "relu", "exp", "sigmoid",
    "tanh", "neg", "badd_col", "bmul_col", "badd_row", "bmul_row",
    "transpose", "reshape", "rowsum", "rowmax", "matmul_bf16", "opaque_copy",
    "tuple", "concat",
)


@dataclass
class Value:
    vid: int
    is_input: bool
    shape: tuple
    dtype: str = "f32"          # "f32" or "bf16"
    op: str | None = None
    args: tuple = ()
    attrs: tuple = ()
    init: tuple = ("uniform", -1.0, 1.0)   # input distribution


@dataclass
class GraphSpec:
    """A dataflow graph in creation (= topological) order.

    Value ids are assigned in creation order to inputs and operator outputs
    alike; the i-th operator created is node i.
    """
    name: str = "graph"
    values: list = field(default_factory=list)
    outputs: list = field(default_factory=list)

    # -- construction -----------------------------------------------------
    def input(self, shape, dtype="f32", init=("uniform", -1.0, 1.0)) -> int:
        v = Value(len(self.values), True, tuple(int(s) for s in shape), dtype, init=init)
        self.values.append(v)
        return v.vid

    def op(self, name, args, attrs=()) -> int:
        assert name in OPS, name
        args = tuple(int(a) for a in args)
        shp = self._shape_of(name, args, attrs)
        v = Value(len(self.values), False, shp, "f32", name, args, tuple(float(a) for a in attrs))
        self.values.append(v)
        return v.vid

    def mark_output(self, vid) -> None:
        if vid not in self.outputs:
            self.outputs.append(int(vid))

    # Shape bookkeeping for graph construction only.
    def _shape_of(self, name, args, attrs):
        s = [self.values[a].shape for a in args]
        if name in ("badd_col", "bmul_col", "badd_row", "bmul_row"):
            return s[0]
        if name == "transpose":
            return (s[0][1], s[0][0])
        if name == "reshape":
            return (int(attrs[0]), int(attrs[1]))
        if name in ("rowsum", "rowmax"):
            return (s[0][0],)
        if name == "tuple":            # its fields stacked by rows
            return (sum(x[0] for x in s), s[0][1])
        if name == "matmul_bf16":
            ta, tb = int(attrs[0]), int(attrs[1])
            m = s[0][1] if ta else s[0][0]
            n = s[1][0] if tb else s[1][1]
            return (m, n)
        return s[0]

    # -- queries ------------------------------------------------------------
    @property
    def inputs(self):
        return [v.vid for v in self.values if v.is_input]

    @property
    def ops(self):
        return [v for v in self.values if not v.is_input]

    def node_of_value(self):
        out, n = {}, 0
        for v in self.values:
            if not v.is_input:
                out[v.vid] = n
                n += 1
        return out

    def consumers(self):
        cons = {v.vid: [] for v in self.values}
        for v in self.values:
            if not v.is_input:
                for a in v.args:
                    cons[a].append(v.vid)
        return cons


def _nbytes(v: Value) -> int:
    return int(np.prod(v.shape)) * (2 if v.dtype == "bf16" else 4)


# ---------------------------------------------------------------------------
# Inputs
# ---------------------------------------------------------------------------

def make_input(spec: GraphSpec, vid: int, seed: int = 0) -> np.ndarray:
    """Draw input `vid` from its distribution with a per-input seeded stream.

    bf16 inputs are returned as float32 arrays whose values are exactly
    representable in bfloat16: the float32 draw has its low 16 bits cleared
    (round toward zero).  The caller converts them to a bf16 tensor exactly.
    """
    v = spec.values[vid]
    assert v.is_input
    rng = np.random.default_rng([seed, vid])
    kind = v.init[0]
    if kind == "uniform":
        a = rng.uniform(v.init[1], v.init[2], size=v.shape)
    elif kind == "normal":
        a = rng.normal(v.init[1], v.init[2], size=v.shape)
    else:
        raise ValueError(kind)
    a = a.astype(np.float32)
    if v.dtype == "bf16":
        a = (a.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    return a


def make_inputs(spec: GraphSpec, seed: int = 0) -> dict:
    return {vid: make_input(spec, vid, seed) for vid in spec.inputs}


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def rnnlm_chain(R=64, C=1024) -> GraphSpec:
    """Mul1 -> Mul2 (broadcast weight) -> row sum -> Sigmoid (DisCo Fig. 2)."""
    g = GraphSpec("rnnlm_chain")
    x = g.input((R, C))
    y = g.input((R, C))
    w = g.input((C,))
    a = g.op("mul", (x, y))
    b = g.op("bmul_col", (a, w))
    s = g.op("rowsum", (b,))
    o = g.op("sigmoid", (s,))
    g.mark_output(o)
    return g


def diamond(R=8192, C=4096) -> GraphSpec:
    """P = X + bias; relu(P), exp(0.01 P), P*Z reconverge in a 3-way add,
    then transpose (TVM FuseOps > Algorithm, the diamond)."""
    g = GraphSpec("diamond")
    x = g.input((R, C))
    bias = g.input((C,))
    z = g.input((R, C))
    p = g.op("badd_col", (x, bias))
    r1 = g.op("relu", (p,))
    t = g.op("scale", (p,), (0.01,))
    r2 = g.op("exp", (t,))
    r3 = g.op("mul", (p, z))
    s = g.op("add", (r1, r2, r3))
    o = g.op("transpose", (s,))
    g.mark_output(o)
    return g


def sf_update(B=512, M=4096, N=4096, lr=0.01, wd=1e-4) -> GraphSpec:
    """G = U^T V (U [B,M], V [B,N] bf16) then W - lr*(G/B + wd*W)."""
    g = GraphSpec("sf_update")
    u = g.input((B, M), "bf16", ("normal", 0.0, 1.0))
    v = g.input((B, N), "bf16", ("normal", 0.0, 1.0))
    w = g.input((M, N), "f32", ("normal", 0.0, 0.02))
    gm = g.op("matmul_bf16", (u, v), (1, 0))
    t1 = g.op("scale", (gm,), (1.0 / B,))
    t2 = g.op("scale", (w,), (wd,))
    t3 = g.op("add", (t1, t2))
    t4 = g.op("scale", (t3,), (lr,))
    o = g.op("sub", (w, t4))
    g.mark_output(o)
    return g


def tensor_fusion_sizes(seed=0, n=161, total=25_600_000, lo=256, hi=2_400_000):
    """Element counts of the gradient set: log-uniform in [lo, hi], then
    rescaled so the counts sum to `total` (clamped to [lo, hi])."""
    rng = np.random.default_rng(seed)
    raw = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    sz = np.clip(np.rint(raw * (total / raw.sum())), lo, hi).astype(np.int64)
    resid = int(total - sz.sum())
    order = np.argsort(-sz, kind="stable")
    i = 0
    while resid != 0:
        j = order[i % n]
        step = min(resid, hi - sz[j]) if resid > 0 else max(resid, lo - sz[j])
        sz[j] += step
        resid -= step
        i += 1
        if i > 10 * n:
            raise RuntimeError("cannot place residual")
    return sz


def tensor_fusion_inputs(sizes, seed=0, std=1e-3):
    """Gradient values ~N(0, std), one seeded stream per tensor."""
    return [np.random.default_rng([seed, 1000 + i]).normal(0.0, std, int(s)).astype(np.float32)
            for i, s in enumerate(sizes)]


def random_dag(seed=0, n_ops=200, R=8192, C=4096, nominal_C=None, nominal_R=None) -> GraphSpec:
    """Seeded random DAG over [R,C], [C,R], [R] and [C] values.

    Categories: elementwise 0.50, broadcast 0.20, injective 0.15, reduce 0.15.
    Operands come from the 16 most recent values.  An interval bound per value
    keeps results finite: exp only on operands bounded by 20, products bounded
    by 1e6.  The topology depends only on the seed; bounds use the nominal
    sizes, so a scaled-down instance has the same graph as the full one.
    """
    assert R != C, "the two 2-D shapes must differ"
    nC = C if nominal_C is None else nominal_C
    nR = R if nominal_R is None else nominal_R
    rng = np.random.default_rng(seed)
    g = GraphSpec(f"random_dag_s{seed}")
    A, Bs = (R, C), (C, R)
    bound = {}
    nominal_cols = {A: nC, Bs: nR}

    def new_input(shape):
        vid = g.input(shape)
        bound[vid] = 1.0
        return vid

    for _ in range(4):
        new_input(A)

    def recent(pred=None):
        cand = [v.vid for v in g.values[-16:] if pred is None or pred(g.values[v.vid])]
        return cand

    def pick(c):
        return int(c[rng.integers(len(c))])

    def any_2d_recent():
        c = recent(lambda v: len(v.shape) == 2)
        if not c:
            c = [v.vid for v in g.values if len(v.shape) == 2]
        return pick(c)

    def same_shape(shape, exclude):
        c = [v for v in recent(lambda v: v.shape == shape) if v != exclude]
        if not c:
            c = [v.vid for v in g.values if v.shape == shape and v.vid != exclude]
        if not c:
            return new_input(shape)
        return pick(c)

    cats = ("ew", "bc", "inj", "red")
    for _ in range(n_ops):
        cat = cats[rng.choice(4, p=[0.5, 0.2, 0.15, 0.15])]
        if cat == "ew":
            prim = pick(recent())
            shape = g.values[prim].shape
            fn = ("add", "mul", "relu", "exp", "sigmoid", "tanh")[rng.integers(6)]
            if fn == "add":
                arity = 2 + int(rng.integers(2))
                ops = [prim] + [same_shape(shape, prim) for _ in range(arity - 1)]
                vid = g.op("add", ops)
                bound[vid] = sum(bound[o] for o in ops)
            elif fn == "mul":
                other = same_shape(shape, prim)
                if bound[prim] * bound[other] > 1e6:
                    vid = g.op("add", (prim, other))
                    bound[vid] = bound[prim] + bound[other]
                else:
                    vid = g.op("mul", (prim, other))
                    bound[vid] = bound[prim] * bound[other]
            else:
                if fn == "exp" and bound[prim] > 20.0:
                    fn = ("relu", "sigmoid", "tanh")[rng.integers(3)]
                vid = g.op(fn, (prim,))
                if fn == "relu":
                    bound[vid] = bound[prim]
                elif fn == "exp":
                    bound[vid] = math.exp(bound[prim])
                else:
                    bound[vid] = 1.0
        elif cat == "bc":
            x = any_2d_recent()
            shape = g.values[x].shape
            vlen = shape[1]
            fn = "badd_col" if rng.random() < 0.75 else "bmul_col"
            if rng.random() < 0.5:
                vec = new_input((vlen,))
            else:
                c = [v.vid for v in g.values if v.shape == (vlen,)]
                vec = pick(c) if c else new_input((vlen,))
            if fn == "bmul_col" and bound[x] * bound[vec] > 1e6:
                fn = "badd_col"
            vid = g.op(fn, (x, vec))
            bound[vid] = bound[x] + bound[vec] if fn == "badd_col" else bound[x] * bound[vec]
        elif cat == "inj":
            x = any_2d_recent()
            shape = g.values[x].shape
            if rng.random() < 0.5:
                vid = g.op("transpose", (x,))
            else:
                vid = g.op("reshape", (x,), (shape[1], shape[0]))
            bound[vid] = bound[x]
        else:
            x = any_2d_recent()
            shape = g.values[x].shape
            if rng.random() < 0.5:
                vid = g.op("rowsum", (x,))
                bound[vid] = bound[x] * nominal_cols[shape]
            else:
                vid = g.op("rowmax", (x,))
                bound[vid] = bound[x]
    cons = g.consumers()
    for v in g.values:
        if not v.is_input and not cons[v.vid]:
            g.mark_output(v.vid)
    return g


def algorithmic_bytes_unfused(spec: GraphSpec) -> int:
    """Bytes an op-by-op execution moves: every op reads its operands and
    writes its output once."""
    tot = 0
    for v in spec.ops:
        tot += sum(_nbytes(spec.values[a]) for a in v.args) + _nbytes(v)
    return tot


CONFIGS = {
    "rnnlm_chain": dict(full=dict(R=64, C=1024), small=dict(R=64, C=1024)),
    "diamond": dict(full=dict(R=8192, C=4096), small=dict(R=200, C=132)),
    "sf_update": dict(full=dict(B=512, M=4096, N=4096), small=dict(B=128, M=256, N=512)),
    "random_dag": dict(full=dict(R=8192, C=4096),
                       small=dict(R=96, C=48, nominal_R=8192, nominal_C=4096)),
}
