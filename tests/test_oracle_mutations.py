"""The pins bite: each test plants a plausible mistake in the oracle (on the
CPU, via monkeypatch) and checks that one of the pins then fails."""
import numpy as np
import pytest

import oracle.kinds as K
import oracle.postdom as PD
import oracle.partition as P
import oracle.execute as E
import oracle.pack as PK
from tests import test_oracle_partition as TP
from tests import test_oracle_postdom as TD
from tests import test_oracle_pack as TK
from tests import test_oracle_execute as TE


def _fails(fn):
    with pytest.raises(AssertionError):
        fn()


def test_mutation_edge_kind_without_broadcast_exception(monkeypatch):
    monkeypatch.setattr(K, "edge_kind", lambda spec, u, v: K.op_kind(spec.values[v].op))
    monkeypatch.setattr(PD, "edge_kind", lambda spec, u, v: K.op_kind(spec.values[v].op))
    _fails(TP.test_matmul_bias_relu_one_group)


def test_mutation_outputs_not_roots(monkeypatch):
    orig = PD.ForwardGraph.__init__

    def init(self, spec):
        orig(self, spec)
        self.to_exit = [not s for s in self.succ]
    monkeypatch.setattr(PD.ForwardGraph, "__init__", init)
    _fails(TD.test_graph_output_is_always_a_root)


def test_mutation_lca_takes_first_consumer(monkeypatch):
    def bad_ipdom(fg):
        par = [(-1 if fg.to_exit[i] else fg.succ[i][0]) for i in range(fg.n)]
        return par, [0] * fg.n
    monkeypatch.setattr(PD, "ipdom", bad_ipdom)
    _fails(TD.test_diamond_from_the_page)


def test_mutation_reduce_initiates(monkeypatch):
    monkeypatch.setattr(P, "K_COMM_REDUCE", -99)
    _fails(TP.test_reduce_is_a_sink_only)


def test_mutation_no_size_limit(monkeypatch):
    monkeypatch.setattr(P.Options.__init__, "__defaults__", (10 ** 9, 64, False))
    _fails(TP.test_max_fused_ops_256)


def test_mutation_bf16_truncates(monkeypatch):
    monkeypatch.setattr(PK, "bf16_rne_bits",
                        lambda x: (np.asarray(x, np.float32).reshape(-1).view(np.uint32) >> 16).astype(np.uint16))
    _fails(TK.test_bf16_rne_golden)


def test_mutation_layout_unaligned(monkeypatch):
    monkeypatch.setattr(PK, "align_up", lambda x, a: x)
    _fails(TK.test_layout_golden)


def test_mutation_add3_single_rounding(monkeypatch):
    orig = E.apply_op

    def bad(op, args, attrs):
        if op == "add" and len(args) == 3:
            return sum(np.asarray(a, np.float64) for a in args).astype(np.float32)
        return orig(op, args, attrs)
    monkeypatch.setattr(E, "apply_op", bad)
    _fails(TE.test_add3_is_two_rounded_adds)


def test_mutation_matmul_ignores_transpose_flag(monkeypatch):
    orig = E.apply_op

    def bad(op, args, attrs):
        if op == "matmul_bf16":
            return orig(op, args, (0, attrs[1])) if args[0].shape[0] == args[1].shape[0] else orig(op, args, attrs)
        return orig(op, args, attrs)
    monkeypatch.setattr(E, "apply_op", bad)
    with pytest.raises((AssertionError, ValueError)):
        TE.test_matmul_equals_sum_of_outer_products()
