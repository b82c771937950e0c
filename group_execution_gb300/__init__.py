"""Fused operator-group execution and tensor-fusion packing on one GB300.

A thin Python layer over libgroupexec.so (C ABI in include/groupexec.h):

* ``Graph``  -- build a dataflow graph of operators (node i = i-th operator);
* ``Plan``   -- FuseOps-style grouping of a graph, one CUDA kernel per group
                (``launch_group``) or per operator (``launch_unfused``);
* ``TensorFusion`` -- pack many float32 gradients into one bf16 fusion buffer
                and unpack them again, one kernel each.

PyTorch supplies device memory and streams only; every step runs in the
library's kernels.  There is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C

from . import _lib
from ._lib import FgError, OPCODES, EXEC_KINDS, FG_F32, FG_BF16  # noqa: F401

__all__ = ["Graph", "Plan", "Partition", "TensorFusion", "FgError", "OPCODES", "graph_from_spec", "plan_threshold",
           "merge_buckets", "simulate"]


def _i32a(xs):
    return (C.c_int32 * max(1, len(xs)))(*xs)


def _stream_handle(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


class Graph:
    def __init__(self):
        self.lib = _lib.load()
        self.h = C.c_void_p()
        _lib.check(self.lib.fg_graph_create(C.byref(self.h)))
        self.shapes = []
        self.dtypes = []

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.fg_graph_destroy(h)
            self.h = None

    def input(self, shape, dtype="f32") -> int:
        dt = FG_BF16 if dtype == "bf16" else FG_F32
        shp = (C.c_int64 * len(shape))(*shape)
        vid = C.c_int32()
        _lib.check(self.lib.fg_graph_add_input(self.h, dt, len(shape), shp, C.byref(vid)))
        self.shapes.append(tuple(shape))
        self.dtypes.append(dtype)
        return vid.value

    def op(self, name, args, attrs=()) -> int:
        vid = C.c_int32()
        at = (C.c_float * max(1, len(attrs)))(*attrs)
        _lib.check(self.lib.fg_graph_add_op(self.h, OPCODES[name], len(args), _i32a(args), len(attrs), at,
                                            C.byref(vid)))
        dt, nd, shp = C.c_int32(), C.c_int32(), (C.c_int64 * 2)()
        _lib.check(self.lib.fg_graph_value_info(self.h, vid.value, C.byref(dt), C.byref(nd), shp))
        self.shapes.append((shp[0],) if nd.value == 1 else (shp[0], shp[1]))
        self.dtypes.append("f32")
        return vid.value

    def mark_output(self, vid):
        _lib.check(self.lib.fg_graph_mark_output(self.h, vid))

    def build(self, max_fused_ops=256, max_args=64, allow_reduce_epilogue=False, wait_limit_ns=2_000_000_000,
              flags=0):
        return Plan(self, max_fused_ops, max_args, allow_reduce_epilogue, wait_limit_ns, flags)

    def partition(self, from_fuseops=True, max_fused_ops=256, max_args=64, allow_reduce_epilogue=False,
                  wait_limit_ns=2_000_000_000, flags=0, patterns=None):
        """An explicit partition to change with fusion moves (Partition.fuse),
        from the FuseOps grouping, singletons, or operator-chain patterns."""
        return Partition(self, from_fuseops, max_fused_ops, max_args, allow_reduce_epilogue, wait_limit_ns, flags,
                         patterns)


def _opts(lib, max_fused_ops, max_args, allow_reduce_epilogue, wait_limit_ns, flags):
    o = _lib.BuildOpts()
    lib.fg_build_opts_default(C.byref(o))
    o.max_fused_ops, o.max_args = max_fused_ops, max_args
    o.allow_reduce_epilogue = int(bool(allow_reduce_epilogue))
    o.wait_limit_ns = wait_limit_ns
    o.flags = flags
    return o


class Partition:
    """Explicit fusion moves (DisCo: an operator fused with one of its
    predecessors, by duplicate or non-duplicate fusion)."""

    def __init__(self, graph, from_fuseops=True, max_fused_ops=256, max_args=64, allow_reduce_epilogue=False,
                 wait_limit_ns=2_000_000_000, flags=0, patterns=None):
        """patterns: list of (name, [op names], private) in priority order
        (FuseOpsByPattern); then from_fuseops is ignored and match_of lists
        the pattern index per operator."""
        self.lib = graph.lib
        self.graph = graph
        o = _opts(self.lib, max_fused_ops, max_args, allow_reduce_epilogue, wait_limit_ns, flags)
        self.h = C.c_void_p()
        self.match_of = None
        if patterns is None:
            _lib.check(self.lib.fg_partition_create(graph.h, C.byref(o), int(bool(from_fuseops)), C.byref(self.h)))
        else:
            codes = [(C.c_int32 * len(ch))(*[OPCODES[x] for x in ch]) for _, ch, _ in patterns]
            arr = (_lib.Pattern * max(1, len(patterns)))(
                *[_lib.Pattern(len(ch), C.cast(cd, C.c_void_p), int(bool(pv))) for (_, ch, pv), cd in zip(patterns, codes)])
            mo = (C.c_int32 * max(1, len(graph.shapes)))()
            _lib.check(self.lib.fg_partition_from_patterns(graph.h, C.byref(o), len(patterns), arr, C.byref(self.h), mo))
            n = C.c_int32()
            _lib.check(self.lib.fg_partition_query(self.h, C.byref(n), None, None))
            self.match_of = list(mo)[:n.value]

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.fg_partition_destroy(h)
            self.h = None

    def fuse(self, node, pred, duplicate=False):
        _lib.check(self.lib.fg_partition_fuse(self.h, node, pred, int(bool(duplicate))))

    def query(self):
        """(group_of, clone_of) per operator, copies included."""
        n = C.c_int32()
        _lib.check(self.lib.fg_partition_query(self.h, C.byref(n), None, None))
        g, c = (C.c_int32 * n.value)(), (C.c_int32 * n.value)()
        _lib.check(self.lib.fg_partition_query(self.h, None, g, c))
        return list(g), list(c)

    def build(self):
        return Plan(self.graph, _handle=self._build_handle())

    def _build_handle(self):
        h = C.c_void_p()
        _lib.check(self.lib.fg_build_from_partition(self.h, C.byref(h)))
        return h


def graph_from_spec(spec) -> Graph:
    """A Graph with the same values, in the same order, as a workloads.GraphSpec."""
    g = Graph()
    for v in spec.values:
        if v.is_input:
            g.input(v.shape, v.dtype)
        else:
            g.op(v.op, v.args, v.attrs)
    for o in spec.outputs:
        g.mark_output(o)
    return g


class GroupInfo:
    def __init__(self, nodes, leaves, out, kind, alg_bytes, alg_flops, status, outs=None):
        self.nodes, self.leaves, self.out = nodes, leaves, out
        self.kind, self.alg_bytes, self.alg_flops, self.status = kind, alg_bytes, alg_flops, status
        self.outs = outs if outs is not None else [out]   # sink output first, then extra outputs

    def __repr__(self):
        return (f"GroupInfo(nodes={self.nodes}, leaves={self.leaves}, out={self.out}, kind={self.kind}, "
                f"alg_bytes={self.alg_bytes})")


class Plan:
    def __init__(self, graph: Graph, max_fused_ops=256, max_args=64, allow_reduce_epilogue=False,
                 wait_limit_ns=2_000_000_000, flags=0, _handle=None):
        self.lib = graph.lib
        self.graph = graph
        if _handle is not None:
            self.h = _handle
        else:
            o = _opts(self.lib, max_fused_ops, max_args, allow_reduce_epilogue, wait_limit_ns, flags)
            self.h = C.c_void_p()
            _lib.check(self.lib.fg_build_groups(graph.h, C.byref(o), C.byref(self.h)))
        nn, ng = C.c_int32(), C.c_int32()
        _lib.check(self.lib.fg_plan_query(self.h, C.byref(nn), C.byref(ng), None, None))
        self.n_nodes, self.n_groups = nn.value, ng.value
        gof, ipd = (C.c_int32 * nn.value)(), (C.c_int32 * nn.value)()
        _lib.check(self.lib.fg_plan_query(self.h, None, None, gof, ipd))
        self.group_of, self.ipdom = list(gof), list(ipd)
        self.groups = [self._info(g) for g in range(self.n_groups)]

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.fg_plan_destroy(h)
            self.h = None

    def _info(self, gid):
        nn, nl = C.c_int32(), C.c_int32()
        self.lib.fg_plan_group_info(self.h, gid, C.byref(nn), None, C.byref(nl), None, None, None, None, None)
        nodes, leaves = (C.c_int32 * max(1, nn.value))(), (C.c_int32 * max(1, nl.value))()
        out, kind, ab, af = C.c_int32(), C.c_int32(), C.c_int64(), C.c_int64()
        st = self.lib.fg_plan_group_info(self.h, gid, C.byref(nn), nodes, C.byref(nl), leaves, C.byref(out),
                                         C.byref(kind), C.byref(ab), C.byref(af))
        no = C.c_int32()
        self.lib.fg_plan_group_outputs(self.h, gid, C.byref(no), None)
        outs = (C.c_int32 * no.value)()
        self.lib.fg_plan_group_outputs(self.h, gid, None, outs)
        return GroupInfo(list(nodes)[:nn.value], list(leaves)[:nl.value], out.value, EXEC_KINDS[kind.value],
                         ab.value, af.value, st, list(outs))

    def exec_info(self, gid):
        v = [C.c_int32() for _ in range(6)]
        _lib.check(self.lib.fg_plan_group_exec_info(self.h, gid, *[C.byref(x) for x in v]))
        return dict(zip(("tile_rows", "tile_cols", "stages", "n_staged", "n_gathered", "prog_len"),
                        [x.value for x in v]))

    def direct_info(self, gid):
        """Whether group gid runs on the direct kernel, its warps per frame
        row, and whether its launch always may begin early."""
        v = [C.c_int32() for _ in range(3)]
        _lib.check(self.lib.fg_plan_group_direct_info(self.h, gid, *[C.byref(x) for x in v]))
        return dict(zip(("direct", "segments", "early_launch"), [x.value for x in v]))

    def source(self, gid):
        """CUDA source the plan compiles for group gid."""
        n = C.c_int64()
        _lib.check(self.lib.fg_plan_group_source(self.h, gid, None, 0, C.byref(n)))
        buf = C.create_string_buffer(n.value + 1)
        _lib.check(self.lib.fg_plan_group_source(self.h, gid, buf, n.value + 1, C.byref(n)))
        return buf.value.decode()

    def _ptrs(self, tensors):
        n = len(self.graph.shapes)
        arr = (C.c_void_p * n)()
        for vid, t in tensors.items():
            arr[vid] = t if isinstance(t, int) else t.data_ptr()
        return arr

    def launch_group(self, gid, tensors, stream=None):
        """tensors: {value id: device tensor or pointer} for the group's leaves and output."""
        _lib.check(self.lib.fg_launch_group(self.h, gid, self._ptrs(tensors), _stream_handle(stream)))

    def launch_unfused(self, node, tensors, stream=None):
        _lib.check(self.lib.fg_launch_unfused(self.h, node, self._ptrs(tensors), _stream_handle(stream)))

    def launch_group_ptrs(self, gid, ptr_array, stream_handle):
        """Pre-marshalled launch (ctypes pointer array indexed by value id)."""
        return self.lib.fg_launch_group(self.h, gid, ptr_array, stream_handle)

    def sync(self, stream=None):
        _lib.check(self.lib.fg_sync_status(self.h, _stream_handle(stream)))


class TensorFusion:
    """Layout of float32 gradient tensors inside one fusion buffer."""

    def __init__(self, grads, buf_dtype="bf16", align=256):
        self.lib = _lib.load()
        n = len(grads)
        numel = (C.c_int64 * n)(*[g.numel() for g in grads])
        ptrs = (C.c_void_p * n)(*[g.data_ptr() for g in grads])
        offs = (C.c_int64 * n)()
        total = C.c_int64()
        self.h = C.c_void_p()
        _lib.check(self.lib.tf_layout_create(n, numel, ptrs, FG_BF16 if buf_dtype == "bf16" else FG_F32, align,
                                             C.byref(self.h), offs, C.byref(total)))
        self.grads = grads
        self.offsets = list(offs)
        self.total_bytes = total.value

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.tf_layout_destroy(h)
            self.h = None

    def pack(self, scale, buf, stream=None):
        _lib.check(self.lib.tf_pack(self.h, C.c_float(scale), C.c_void_p(buf.data_ptr()), _stream_handle(stream)))

    def unpack(self, uscale, buf, stream=None):
        _lib.check(self.lib.tf_unpack(self.h, C.c_float(uscale), C.c_void_p(buf.data_ptr()),
                                      _stream_handle(stream)))

    def sync(self, stream=None):
        """Waits for the stream; raises FgError (FG_ETIMEOUT) if an unpack
        recorded an expired wait."""
        _lib.check(self.lib.tf_sync_status(self.h, _stream_handle(stream)))

    def pack_range(self, first, count, scale, buf, stream=None):
        """Pack tensors first .. first+count-1 only (e.g. one bucket)."""
        _lib.check(self.lib.tf_pack_range(self.h, first, count, C.c_float(scale), C.c_void_p(buf.data_ptr()),
                                          _stream_handle(stream)))

    def unpack_range(self, first, count, uscale, buf, stream=None):
        _lib.check(self.lib.tf_unpack_range(self.h, first, count, C.c_float(uscale), C.c_void_p(buf.data_ptr()),
                                            _stream_handle(stream)))

    def set_buckets(self, bounds):
        """Bucket table for one-launch packing: bucket b holds tensors
        bounds[b] .. bounds[b+1]-1 (as plan_threshold returns them)."""
        nb = len(bounds) - 1
        arr = (C.c_int32 * len(bounds))(*[int(x) for x in bounds])
        _lib.check(self.lib.tf_layout_set_buckets(self.h, nb, arr))

    def pack_buckets(self, scale, buf, stream=None):
        """Pack every tensor in one launch; each bucket is marked ready as
        soon as its bytes are written (see bucket_wait)."""
        _lib.check(self.lib.tf_pack_buckets(self.h, C.c_float(scale), C.c_void_p(buf.data_ptr()),
                                            _stream_handle(stream)))

    def pack_buckets_observed(self, scale, buf, times, seq_offset=0, wait_limit_ns=100_000_000, stream=None):
        """pack_buckets with one more CTA in the launch that watches the
        buckets' counts: times (int64 device tensor, n_buckets + 1)
        receives when each bucket was seen ready (device global timer, ns)
        and, last, when the packing CTAs finished."""
        _lib.check(self.lib.tf_pack_buckets_observed(self.h, C.c_float(scale), C.c_void_p(buf.data_ptr()),
                                                     C.c_void_p(times.data_ptr()), seq_offset, wait_limit_ns,
                                                     _stream_handle(stream)))

    def bucket_wait(self, b, stream=None):
        """Make `stream` wait until bucket b of the last pack_buckets launch
        is ready (a stream-ordered wait: no kernel runs for it)."""
        _lib.check(self.lib.tf_bucket_wait(self.h, b, _stream_handle(stream)))

    def bucket_ready(self, b):
        """True once bucket b of the last pack_buckets launch is written
        (a synchronous read of its count)."""
        r = C.c_int32()
        _lib.check(self.lib.tf_bucket_ready(self.h, b, C.byref(r)))
        return bool(r.value)

    def bucket_ranges(self, bounds):
        """Byte range [start, end) of every bucket in the fusion buffer."""
        starts = [self.offsets[b] if b < len(self.offsets) else self.total_bytes for b in bounds]
        return [(starts[k], starts[k + 1]) for k in range(len(bounds) - 1)]


def layout_offsets(numels, buf_dtype="bf16", align=256):
    """Byte offsets of the tensors in the fusion buffer and its total size,
    computed on the host (no device): as TensorFusion lays them out."""
    lib = _lib.load()
    n = len(numels)
    arr = (C.c_int64 * max(n, 1))(*[int(x) for x in numels])
    offs = (C.c_int64 * max(n, 1))()
    total = C.c_int64()
    _lib.check(lib.tf_layout_offsets(n, arr, FG_BF16 if buf_dtype == "bf16" else FG_F32, align, offs,
                                     C.byref(total)))
    return list(offs[:n]), total.value


def plan_threshold(numels, threshold_bytes, buf_dtype="bf16", align=256):
    """Threshold fusion of gradient tensors (in production order) into
    AllReduce buckets; returns the boundaries: bucket b holds tensors
    bounds[b] .. bounds[b+1]-1.  Host only."""
    lib = _lib.load()
    n = len(numels)
    arr = (C.c_int64 * max(n, 1))(*[int(x) for x in numels])
    bounds = (C.c_int32 * (n + 1))()
    nb = C.c_int32()
    _lib.check(lib.tf_plan_threshold(n, arr, FG_BF16 if buf_dtype == "bf16" else FG_F32, align, threshold_bytes,
                                     bounds, C.byref(nb)))
    return list(bounds[:nb.value + 1])


def merge_buckets(bounds, j):
    """Bucket j combined with its neighbour j+1."""
    lib = _lib.load()
    arr = (C.c_int32 * len(bounds))(*bounds)
    nb = C.c_int32(len(bounds) - 1)
    _lib.check(lib.tf_buckets_merge(arr, C.byref(nb), j))
    return list(arr[:nb.value + 1])


def simulate(op_time, edges, tensor_producer, tensor_bytes, buckets, c, d, ar_edges=()):
    """Training-step time from the library's simulator (fg_simulate): op_time
    per operator, edges (src, dst), gradient tensors (producer, bytes),
    buckets (lists of tensor ids, one AllReduce each), AllReduce time
    c * bytes + d, ar_edges (bucket, operator).  Returns (total, op_finish,
    ar_start, ar_finish)."""
    lib = _lib.load()
    n, nt, nb = len(op_time), len(tensor_producer), len(buckets)

    def arr(ctype, xs):
        return (ctype * max(1, len(xs)))(*xs)

    keep = [arr(C.c_double, [float(x) for x in op_time]), arr(C.c_int32, [int(a) for a, _ in edges]),
            arr(C.c_int32, [int(b) for _, b in edges]), arr(C.c_int32, [int(x) for x in tensor_producer]),
            arr(C.c_double, [float(x) for x in tensor_bytes])]
    bounds = [0]
    flat = []
    for bk in buckets:
        flat += [int(x) for x in bk]
        bounds.append(len(flat))
    keep += [arr(C.c_int32, bounds), arr(C.c_int32, flat), arr(C.c_int32, [int(b) for b, _ in ar_edges]),
             arr(C.c_int32, [int(t) for _, t in ar_edges])]
    pr = _lib.SimProblem(n, C.cast(keep[0], C.c_void_p), len(edges), C.cast(keep[1], C.c_void_p),
                         C.cast(keep[2], C.c_void_p), nt, C.cast(keep[3], C.c_void_p), C.cast(keep[4], C.c_void_p),
                         nb, C.cast(keep[5], C.c_void_p), C.cast(keep[6], C.c_void_p), float(c), float(d),
                         len(ar_edges), C.cast(keep[7], C.c_void_p), C.cast(keep[8], C.c_void_p))
    total = C.c_double()
    fin, s0, f0 = (C.c_double * max(1, n))(), (C.c_double * max(1, nb))(), (C.c_double * max(1, nb))()
    _lib.check(lib.fg_simulate(C.byref(pr), C.byref(total), fin, s0, f0))
    return total.value, list(fin)[:n], list(s0)[:nb], list(f0)[:nb]
