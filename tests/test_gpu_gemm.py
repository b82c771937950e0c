"""GPU parity of the GEMM-epilogue kernel (tcgen05 MMA into TMEM, fused
elementwise tail) against the oracle's float64 matmul, through the C ABI."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import execute as OE
from tests._helpers import rel_err, TOL_F32, TOL_BF16
from tests._gpu import prepare, run_fused, run_unfused
from group_execution_gb300 import _lib

pytestmark = pytest.mark.gpu
MODES = [0, _lib.FG_FLAG_INTERPRET]
PAIRS = 1 << 16                        # GEMM cluster shape: CTA pairs (ignored: the only shape)
KB1, KB2 = 1 << 18, 2 << 18            # K blocks per operand ring slot
TN256, TN128 = 1 << 22, 2 << 22        # columns of a pair's tile
KSPLIT = 1 << 20                       # schedule: round robin, the last round's units cut into K pieces
SHAPES = [PAIRS | KB2, PAIRS | KB1, PAIRS | TN128, PAIRS | KB1 | TN128]


def _matmul_graph(K, M, N, ta, tb, epi=None):
    g = W.GraphSpec("mm")
    a = g.input((K, M) if ta else (M, K), "bf16", ("normal", 0.0, 1.0))
    b = g.input((N, K) if tb else (K, N), "bf16", ("normal", 0.0, 1.0))
    m = g.op("matmul_bf16", (a, b), (ta, tb))
    out = m
    if epi == "bias_relu":
        v = g.input((N,))
        out = g.op("relu", (g.op("badd_col", (m, v)),))
    elif epi == "trans_leaf":
        # y2 has two transposed paths into the epilogue, so its post-dominator
        # is the add inside the matmul group and it fuses there (an injective
        # group alone never joins a matmul group)
        y = g.input((N, M))
        y2 = g.op("relu", (y,))
        t1 = g.op("transpose", (y2,))
        t2 = g.op("transpose", (g.op("exp", (y2,)),))
        r = g.input((M,))
        out = g.op("badd_row", (g.op("add", (m, t1, t2)), r))
    g.mark_output(out)
    return g


def _check_matmul_bound(got, A, B):
    """|G - exact| <= K * 2^-22 * sum_k |a_k b_k| elementwise (f32 accumulation
    of exact bf16 products, with slack for the tensor core's adder)."""
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    exact = A64 @ B64
    bound = A64.shape[1] * 2.0 ** -22 * (np.abs(A64) @ np.abs(B64)) + 1e-30
    assert np.all(np.abs(got.astype(np.float64) - exact) <= bound), np.max(np.abs(got - exact) / bound)


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("kmn", [(128, 256, 512), (72, 200, 264), (512, 128, 256), (64, 384, 768)])
@pytest.mark.parametrize("mode", MODES)
def test_matmul_layouts(ta, tb, kmn, mode):
    K, M, N = kmn
    spec = _matmul_graph(K, M, N, ta, tb)
    g, plan, inputs, dev = prepare(spec, flags=mode)
    assert plan.groups[0].kind == "gemm"
    env = run_fused(plan, spec, dev)
    plan.sync()
    got = env[spec.outputs[0]].cpu().numpy()
    A = inputs[0].T if ta else inputs[0]
    B = inputs[1].T if tb else inputs[1]
    _check_matmul_bound(got, A, B)


@pytest.mark.parametrize("epi", ["bias_relu", "trans_leaf"])
@pytest.mark.parametrize("mode", MODES)
def test_matmul_epilogues(epi, mode):
    spec = _matmul_graph(96, 256, 512, 1, 0, epi)
    g, plan, inputs, dev = prepare(spec, flags=mode)
    assert plan.n_groups == 1 and plan.groups[0].kind == "gemm"
    env = run_fused(plan, spec, dev)
    plan.sync()
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    assert rel_err(env[spec.outputs[0]].cpu().numpy(), ref) <= 1e-4


def _sf_update(B, M, N, mode):
    return _sf_update_flags(B, M, N, mode)


def _sf_update_flags(B, M, N, mode):
    spec = W.sf_update(B, M, N)
    g, plan, inputs, dev = prepare(spec, flags=mode)
    assert plan.n_groups == 1 and plan.groups[0].kind == "gemm"
    env = run_fused(plan, spec, dev)
    plan.sync()
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    got = env[spec.outputs[0]].cpu().numpy()
    w = inputs[2]
    assert rel_err(got, ref) <= TOL_F32
    # the update itself, W - W_new, on its own (W_new ~ W hides G errors)
    assert rel_err(w - got, w - ref) <= TOL_BF16
    return plan, spec, dev, env, ref


@pytest.mark.parametrize("mode", MODES)
def test_sf_update_small(mode):
    plan, spec, dev, env, ref = _sf_update(128, 256, 512, mode)
    envu = run_unfused(plan, spec, dev)
    plan.sync()
    assert rel_err(envu[spec.outputs[0]].cpu().numpy(), ref) <= TOL_F32


def test_sf_update_full():
    _sf_update(512, 4096, 4096, 0)


@pytest.mark.parametrize("K,M,N,cap", [(1024, 1024, 1024, 5), (1024, 1024, 1024, 7), (2048, 1024, 1024, 5),
                                       (1088, 768, 1280, 7)])
@pytest.mark.parametrize("kb", [KB2, KB1])
def test_split_tail(K, M, N, cap, kb):
    """The last round's tiles split along K (CTA pairs capped so that a tail
    exists): the partial accumulators meet in the workspace and the last
    piece finishes the epilogue; run twice, so the arrival counters are seen
    to reset."""
    spec = W.sf_update(K, M, N)
    g, plan, inputs, dev = prepare(spec, flags=(cap << 8) | PAIRS | KSPLIT | kb)
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    w = inputs[2]
    for _ in range(2):
        env = run_fused(plan, spec, dev)
        plan.sync()
        got = env[spec.outputs[0]].cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(w - got, w - ref) <= TOL_BF16


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1)])
def test_split_tail_plain_layouts(ta, tb):
    K, M, N = 1024, 1024, 768
    spec = _matmul_graph(K, M, N, ta, tb)
    g, plan, inputs, dev = prepare(spec, flags=(5 << 8) | PAIRS | KSPLIT)
    env = run_fused(plan, spec, dev)
    plan.sync()
    A = inputs[0].T if ta else inputs[0]
    B = inputs[1].T if tb else inputs[1]
    _check_matmul_bound(env[spec.outputs[0]].cpu().numpy(), A, B)


def test_split_tail_full_size():
    # 256 pair tiles on 76 pairs: the last 28 run as K halves
    _sf_update(1024, 4096, 4096, KSPLIT)


def test_column_half_tail_full_size():
    # 256 pair tiles on 76 pairs: the last 28 run as 56 column halves (the
    # default for CTA pairs)
    _sf_update(1024, 4096, 4096, 0)


# ---- ring granularity and tile widths ----

@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("kmn", [(1024, 512, 1024), (1096, 392, 1288), (200, 264, 600), (64, 128, 512)])
@pytest.mark.parametrize("shape", SHAPES)
def test_cluster_shapes_layouts(ta, tb, kmn, shape):
    """One- and two-K-block ring slots and 128-column pair tiles, every
    operand layout; ragged M, N and K, K shorter than one ring slot."""
    K, M, N = kmn
    spec = _matmul_graph(K, M, N, ta, tb)
    g, plan, inputs, dev = prepare(spec, flags=shape)
    env = run_fused(plan, spec, dev)
    plan.sync()
    A = inputs[0].T if ta else inputs[0]
    B = inputs[1].T if tb else inputs[1]
    _check_matmul_bound(env[spec.outputs[0]].cpu().numpy(), A, B)


@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 1)])
@pytest.mark.parametrize("kb", [KB2, KB1])
def test_pairs_stream_k_plain(ta, tb, kb):
    """A plain matmul with pairs capped so that each runs an equal share of
    all units' ring slots (stream-K)."""
    K, M, N = 2048, 1024, 1536
    spec = _matmul_graph(K, M, N, ta, tb)
    g, plan, inputs, dev = prepare(spec, flags=(5 << 8) | PAIRS | (2 << 20) | kb)
    env = run_fused(plan, spec, dev)
    plan.sync()
    A = inputs[0].T if ta else inputs[0]
    B = inputs[1].T if tb else inputs[1]
    _check_matmul_bound(env[spec.outputs[0]].cpu().numpy(), A, B)


@pytest.mark.parametrize("epi", ["bias_relu", "trans_leaf"])
@pytest.mark.parametrize("shape", SHAPES)
def test_cluster_shapes_epilogues(epi, shape):
    spec = _matmul_graph(1024, 256, 1024, 1, 0, epi)
    g, plan, inputs, dev = prepare(spec, flags=shape)
    assert plan.n_groups == 1 and plan.groups[0].kind == "gemm"
    env = run_fused(plan, spec, dev)
    plan.sync()
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    assert rel_err(env[spec.outputs[0]].cpu().numpy(), ref) <= 1e-4


def test_sf_update_k4096_full_size():
    """The compute-bound SF update (B = K = 4096) in the default launch: CTA
    pairs, the last round's units cut into column halves."""
    _sf_update(4096, 4096, 4096, 0)


@pytest.mark.parametrize("K,M,N,cap,kb", [(1024, 1024, 1024, 5, KB2), (1024, 1024, 768, 7, KB1), (1024, 520, 1160, 3, KB2)])
def test_tn128_split_tail(K, M, N, cap, kb):
    """128-column pair tiles with the last round split along K (the workspace
    and flags sized for the narrower tiles); run twice."""
    spec = W.sf_update(K, M, N)
    g, plan, inputs, dev = prepare(spec, flags=(cap << 8) | PAIRS | TN128 | kb)
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    w = inputs[2]
    for _ in range(2):
        env = run_fused(plan, spec, dev)
        plan.sync()
        got = env[spec.outputs[0]].cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(w - got, w - ref) <= TOL_BF16


def test_sf_update_full_tn128():
    """The HBM-bound SF update (K = 512) in 128-column pair tiles."""
    _sf_update_flags(512, 4096, 4096, PAIRS | TN128)


SK = 2 << 20   # schedule: equal shares of all tiles' K steps


@pytest.mark.parametrize("K,M,N,cap,kb", [(2048, 1024, 1024, 5, KB2), (1152, 776, 1800, 7, KB1), (4096, 512, 768, 4, KB2),
                                          (2048, 1024, 2048, 3, KB1), (2048, 1024, 2048, 7, KB2),
                                          (1152, 776, 1800, 6, KB2), (4096, 512, 1024, 3, KB1)])
def test_pairs_stream_k(K, M, N, cap, kb):
    """CTA pairs walking equal shares of all tiles' K steps: a share boundary
    cuts a tile into two pieces, the one ending a share finishing it; run
    twice (the ready flags are cleared by their readers)."""
    spec = W.sf_update(K, M, N)
    g, plan, inputs, dev = prepare(spec, flags=(cap << 8) | PAIRS | SK | kb)
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    w = inputs[2]
    for _ in range(2):
        env = run_fused(plan, spec, dev)
        plan.sync()
        got = env[spec.outputs[0]].cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(w - got, w - ref) <= TOL_BF16


ST_PRODUCER, ST_WARPS = 1 << 24, 2 << 24   # in-place results stored by the leaf producer / by the epilogue warps


@pytest.mark.parametrize("store", [ST_PRODUCER, ST_WARPS])
@pytest.mark.parametrize("K,M,N,extra", [
    (512, 4096, 4096, 0),                                # the HBM-bound update, default launch (six leaf buffers)
    (4096, 1024, 1024, 0),                               # long K: two leaf buffers
    (1024, 1024, 1024, (5 << 8) | PAIRS | KSPLIT | KB2), # last round split along K
    (1024, 1024, 1024, (5 << 8) | PAIRS | KB2),          # last round cut into column halves
    (1024, 520, 1160, (3 << 8) | PAIRS | KSPLIT | KB1),  # ragged rows and columns, split tail
    (1024, 1024, 768, (7 << 8) | PAIRS | TN128 | KB1),   # 128-column pair tiles
    (4096, 512, 768, (4 << 8) | PAIRS | SK | KB2),       # stream-K shares, two leaf buffers
    (512, 776, 1000, (3 << 8) | PAIRS | SK | KB2),       # stream-K shares, ragged
])
def test_inplace_store_modes(store, K, M, N, extra):
    """Results written in place of the IDENT leaf's chunk leave either in one
    copy per 128 x 32 chunk from the leaf producer before it reloads the
    buffer, or in each epilogue warp's copy of its rows, the warp freeing the
    buffer once the copy has read them; every schedule and tile shape, run
    twice (split flags are cleared by readers)."""
    spec = W.sf_update(K, M, N)
    g, plan, inputs, dev = prepare(spec, flags=extra | store)
    assert plan.n_groups == 1 and plan.groups[0].kind == "gemm"
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    w = inputs[2]
    for _ in range(2):
        env = run_fused(plan, spec, dev)
        plan.sync()
        got = env[spec.outputs[0]].cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(w - got, w - ref) <= TOL_BF16


NSPLIT = 3 << 20   # schedule: round robin, the last round's units cut into their column halves


@pytest.mark.parametrize("K,M,N,cap", [
    (512, 1024, 1024, 5),    # one unit cut
    (1024, 1024, 1024, 7),   # two units cut
    (1024, 1024, 1160, 9),   # the second half partly past N
    (1024, 1024, 1088, 9),   # the second half wholly past N
    (256, 520, 1160, 3),     # ragged rows and columns
    (4096, 1024, 1024, 5),   # long K
])
@pytest.mark.parametrize("kb", [KB2, KB1])
def test_column_half_tail(K, M, N, cap, kb):
    """The last round's units cut into their two 128-column halves, each over
    all of K on a pair of its own (half-width B boxes and MMAs, four epilogue
    chunks, no partial sums); run twice."""
    spec = W.sf_update(K, M, N)
    g, plan, inputs, dev = prepare(spec, flags=(cap << 8) | PAIRS | NSPLIT | kb)
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    w = inputs[2]
    for _ in range(2):
        env = run_fused(plan, spec, dev)
        plan.sync()
        got = env[spec.outputs[0]].cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(w - got, w - ref) <= TOL_BF16


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("mode", MODES)
def test_column_half_tail_layouts(ta, tb, mode):
    """Column-half tail units in every operand layout (K-major B takes the
    half-width K-block stride), compiled and interpreted epilogues."""
    K, M, N = 512, 1024, 768
    spec = _matmul_graph(K, M, N, ta, tb)
    g, plan, inputs, dev = prepare(spec, flags=(5 << 8) | PAIRS | NSPLIT | mode)
    env = run_fused(plan, spec, dev)
    plan.sync()
    A = inputs[0].T if ta else inputs[0]
    B = inputs[1].T if tb else inputs[1]
    _check_matmul_bound(env[spec.outputs[0]].cpu().numpy(), A, B)


TN224 = 3 << 22   # 224-column pair tiles (the choice where their rounds come out even)


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("kmn", [(1024, 512, 1024), (1096, 392, 1288), (200, 264, 600), (64, 128, 512),
                                 (512, 256, 4096)])
@pytest.mark.parametrize("kb", [KB2, KB1])
def test_tn224_layouts(ta, tb, kmn, kb):
    """224-column pair tiles: each CTA's B half starts at a multiple of 16
    columns (2-D boxes for an N-contiguous B), the MMAs read 112 of the 128
    staged columns; ragged M, N and K, every operand layout."""
    K, M, N = kmn
    spec = _matmul_graph(K, M, N, ta, tb)
    g, plan, inputs, dev = prepare(spec, flags=TN224 | kb)
    assert "gemm_body<fg::JitEpi, %d, 224>" % (1 if kb == KB1 else 2) in plan.source(0)
    env = run_fused(plan, spec, dev)
    plan.sync()
    A = inputs[0].T if ta else inputs[0]
    B = inputs[1].T if tb else inputs[1]
    _check_matmul_bound(env[spec.outputs[0]].cpu().numpy(), A, B)


@pytest.mark.parametrize("epi", ["bias_relu", "trans_leaf"])
def test_tn224_epilogues(epi):
    spec = _matmul_graph(1024, 512, 1344, 1, 0, epi)
    g, plan, inputs, dev = prepare(spec, flags=TN224)
    env = run_fused(plan, spec, dev)
    plan.sync()
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    assert rel_err(env[spec.outputs[0]].cpu().numpy(), ref) <= TOL_F32


@pytest.mark.parametrize("store", [ST_PRODUCER, ST_WARPS])
@pytest.mark.parametrize("K", [512, 4096])
def test_tn224_sf_update_full_size(store, K):
    """The sufficient-factor update at full size in 224-column tiles (304
    tiles, four rounds on 76 pairs), both in-place store modes, run twice."""
    spec = W.sf_update(K, 4096, 4096)
    g, plan, inputs, dev = prepare(spec, flags=TN224 | store)
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    w = inputs[2]
    for _ in range(2):
        env = run_fused(plan, spec, dev)
        plan.sync()
        got = env[spec.outputs[0]].cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(w - got, w - ref) <= TOL_BF16


RING64, RING96 = 1 << 29, 2 << 29   # operand ring of 64 or 96 KB, the leaf buffers taking the rest


@pytest.mark.parametrize("K,M,N,extra", [
    (512, 1024, 1024, RING96 | KB1),                       # eight leaf buffers; the last item as any other
    (512, 1024, 1024, RING64 | KB2),                       # a single operand slot
    (4096, 1024, 1024, RING96 | KB1),                      # long K: the leaf producer stores in place
    (1024, 1024, 1024, (5 << 8) | KSPLIT | KB1 | RING64),  # split along K: the partial read from global
    (1024, 1024, 1024, (5 << 8) | NSPLIT | KB1 | RING96),  # column halves
    (512, 776, 1000, (3 << 8) | SK | KB2 | RING64),        # stream-K shares, ragged
])
def test_operand_ring_sizes(K, M, N, extra):
    """Operand rings below the size the CTA's last item stages its results in
    (the last item then writes through the leaf buffers like the others);
    every schedule, run twice."""
    spec = W.sf_update(K, M, N)
    g, plan, inputs, dev = prepare(spec, flags=extra)
    assert plan.n_groups == 1 and plan.groups[0].kind == "gemm"
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    w = inputs[2]
    for _ in range(2):
        env = run_fused(plan, spec, dev)
        plan.sync()
        got = env[spec.outputs[0]].cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(w - got, w - ref) <= TOL_BF16


RING64, RING96 = 1 << 29, 2 << 29   # operand ring of 64 or 96 KB, the leaf buffers taking the rest


@pytest.mark.parametrize("K,M,N,extra", [
    (512, 1024, 1024, RING96 | KB1),                       # eight leaf buffers; the last item as any other
    (512, 1024, 1024, RING64 | KB2),                       # a single operand slot
    (4096, 1024, 1024, RING96 | KB1),                      # long K: the leaf producer stores in place
    (1024, 1024, 1024, (5 << 8) | KSPLIT | KB1 | RING64),  # split along K: the partial read from global
    (1024, 1024, 1024, (5 << 8) | NSPLIT | KB1 | RING96),  # column halves
    (512, 776, 1000, (3 << 8) | SK | KB2 | RING64),        # stream-K shares, ragged
])
def test_operand_ring_sizes(K, M, N, extra):
    """Operand rings below the size the CTA's last item stages its results in
    (the last item then writes through the leaf buffers like the others);
    every schedule, run twice."""
    spec = W.sf_update(K, M, N)
    g, plan, inputs, dev = prepare(spec, flags=extra)
    assert plan.n_groups == 1 and plan.groups[0].kind == "gemm"
    ref = OE.run_unfused(spec, inputs)[spec.outputs[0]]
    w = inputs[2]
    for _ in range(2):
        env = run_fused(plan, spec, dev)
        plan.sync()
        got = env[spec.outputs[0]].cpu().numpy()
        assert rel_err(got, ref) <= TOL_F32
        assert rel_err(w - got, w - ref) <= TOL_BF16

