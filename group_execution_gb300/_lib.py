"""ctypes binding of libgroupexec.so (argument marshalling only).

Every entry point of include/groupexec.h is declared here with its C
signature.  There is no Python implementation of anything behind them: if the
library cannot be built or loaded, `load()` raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re
import threading

from . import build as _build

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(HERE), "include", "groupexec.h")

FG_OK, FG_EINVAL, FG_ESHAPE, FG_EUNSUPPORTED, FG_ENOMEM, FG_ECUDA, FG_ETIMEOUT, FG_EDEVICE = range(8)
FG_F32, FG_BF16 = 0, 1
FG_FLAG_INTERPRET = 1 << 26
FG_FLAG_INJECT_NO_LOADS = 1 << 27
FG_FLAG_NO_SMALL = 1 << 28          # small groups too run the pipelined kernels
STATUS_NAMES = ["FG_OK", "FG_EINVAL", "FG_ESHAPE", "FG_EUNSUPPORTED", "FG_ENOMEM", "FG_ECUDA",
                "FG_ETIMEOUT", "FG_EDEVICE"]

OPCODES = {name: i for i, name in enumerate((
    "add", "sub", "mul", "div", "scale", "addc", "relu", "exp", "sigmoid", "tanh", "neg",
    "badd_col", "bmul_col", "badd_row", "bmul_row", "transpose", "reshape", "rowsum", "rowmax",
    "matmul_bf16", "opaque_copy", "tuple", "concat"))}
EXEC_KINDS = ("elementwise", "reduce", "gemm")


class BuildOpts(C.Structure):
    _fields_ = [("max_fused_ops", C.c_int32), ("max_args", C.c_int32),
                ("allow_reduce_epilogue", C.c_int32), ("flags", C.c_int32),
                ("wait_limit_ns", C.c_int64)]


class FgError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES[status] if 0 <= status < 8 else status}: {msg}")
        self.status = status


_P = C.c_void_p
_I32, _I64, _F = C.c_int32, C.c_int64, C.c_float
_PI32, _PI64, _PF = C.POINTER(C.c_int32), C.POINTER(C.c_int64), C.POINTER(C.c_float)

SIGNATURES = {
    "fg_build_opts_default": (None, [C.POINTER(BuildOpts)]),
    "fg_graph_create": (_I32, [C.POINTER(_P)]),
    "fg_graph_add_input": (_I32, [_P, _I32, _I32, _PI64, _PI32]),
    "fg_graph_add_op": (_I32, [_P, _I32, _I32, _PI32, _I32, _PF, _PI32]),
    "fg_graph_mark_output": (_I32, [_P, _I32]),
    "fg_graph_value_info": (_I32, [_P, _I32, _PI32, _PI32, _PI64]),
    "fg_graph_destroy": (None, [_P]),
    "fg_build_groups": (_I32, [_P, C.POINTER(BuildOpts), C.POINTER(_P)]),
    "fg_plan_query": (_I32, [_P, _PI32, _PI32, _PI32, _PI32]),
    "fg_plan_group_info": (_I32, [_P, _I32, _PI32, _PI32, _PI32, _PI32, _PI32, _PI32, _PI64, _PI64]),
    "fg_launch_group": (_I32, [_P, _I32, C.POINTER(_P), _P]),
    "fg_launch_unfused": (_I32, [_P, _I32, C.POINTER(_P), _P]),
    "fg_sync_status": (_I32, [_P, _P]),
    "fg_plan_group_exec_info": (_I32, [_P, _I32, _PI32, _PI32, _PI32, _PI32, _PI32, _PI32]),
    "fg_plan_group_direct_info": (_I32, [_P, _I32, _PI32, _PI32, _PI32]),
    "fg_plan_group_source": (_I32, [_P, _I32, C.c_char_p, _I64, _PI64]),
    "fg_plan_destroy": (None, [_P]),
    "fg_last_error": (C.c_char_p, []),
    "fg_row_reduce_noalloc": (_I32, [_I32, _P, _I64, _I64, _P, _P]),
    "fg_row_reduce_noalloc_status": (_I32, [_P]),
    "tf_layout_create": (_I32, [_I32, _PI64, C.POINTER(_P), _I32, _I64, C.POINTER(_P), _PI64, _PI64]),
    "tf_pack": (_I32, [_P, _F, _P, _P]),
    "tf_layout_offsets": (_I32, [_I32, _PI64, _I32, _I64, _PI64, _PI64]),
    "tf_unpack": (_I32, [_P, _F, _P, _P]),
    "tf_sync_status": (_I32, [_P, _P]),
    "fg_plan_group_outputs": (_I32, [_P, _I32, _P, _P]),
    "fg_partition_create": (_I32, [_P, _P, _I32, _P]),
    "fg_partition_fuse": (_I32, [_P, _I32, _I32, _I32]),
    "fg_partition_from_patterns": (_I32, [_P, _P, _I32, _P, _P, _P]),
    "fg_partition_query": (_I32, [_P, _P, _P, _P]),
    "fg_build_from_partition": (_I32, [_P, _P]),
    "fg_partition_destroy": (None, [_P]),
    "fg_simulate": (_I32, [_P, _P, _P, _P, _P]),
    "tf_plan_threshold": (_I32, [_I32, _P, _I32, _I64, _I64, _P, _P]),
    "tf_buckets_merge": (_I32, [_P, _P, _I32]),
    "tf_pack_range": (_I32, [_P, _I32, _I32, _F, _P, _P]),
    "tf_unpack_range": (_I32, [_P, _I32, _I32, _F, _P, _P]),
    "tf_layout_set_buckets": (_I32, [_P, _I32, _P]),
    "tf_pack_buckets": (_I32, [_P, _F, _P, _P]),
    "tf_pack_buckets_observed": (_I32, [_P, _F, _P, _P, C.c_uint32, _I64, _P]),
    "tf_bucket_wait": (_I32, [_P, _I32, _P]),
    "tf_bucket_ready": (_I32, [_P, _I32, _P]),
    "tf_layout_destroy": (None, [_P]),
}

_lock = threading.Lock()
_handle = None


def header_symbols():
    """Function names declared in include/groupexec.h."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*([a-z_]+)\s*\(", txt, flags=re.M)))


def load(build_if_needed=True):
    """Load (building first if stale) the in-tree libgroupexec.so."""
    global _handle
    with _lock:
        if _handle is not None:
            return _handle
        path = _build.LIB
        if build_if_needed:
            path = _build.build()
        if not os.path.exists(path):
            raise FgError(FG_ECUDA, f"{path} is missing: build it with group_execution_gb300.build.build()")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _handle = lib
        return lib


class Pattern(C.Structure):
    """fg_pattern of groupexec.h."""
    _fields_ = [("n_ops", C.c_int32), ("opcodes", C.c_void_p), ("private_intermediates", C.c_int32)]


class SimProblem(C.Structure):
    """fg_sim_problem of groupexec.h."""
    _fields_ = [("n_ops", C.c_int32), ("op_time", C.c_void_p), ("n_edges", C.c_int32),
                ("edge_src", C.c_void_p), ("edge_dst", C.c_void_p), ("n_tensors", C.c_int32),
                ("tensor_producer", C.c_void_p), ("tensor_bytes", C.c_void_p), ("n_buckets", C.c_int32),
                ("bucket_bounds", C.c_void_p), ("bucket_tensors", C.c_void_p), ("ar_c", C.c_double),
                ("ar_d", C.c_double), ("n_ar_edges", C.c_int32), ("ar_edge_bucket", C.c_void_p),
                ("ar_edge_op", C.c_void_p)]


def check(status):
    if status != FG_OK:
        raise FgError(status, load().fg_last_error().decode())
    return status
