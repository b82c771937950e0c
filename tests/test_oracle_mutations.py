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
from tests import test_oracle_composition as TC


def _fails(fn):
    # an assertion fails, or an expected error is no longer raised
    with pytest.raises((AssertionError, pytest.fail.Exception)):
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


def test_mutation_no_phase2(monkeypatch):
    # tuples never recognised: no phase 2, no absorbed-tuple pattern
    monkeypatch.setattr(P, "K_TUPLE", -99)
    _fails(TP.test_phase1_absorbs_the_tuple_phase2_its_fields)


def test_mutation_absorbed_tuple_keeps_its_pattern(monkeypatch):
    def union_into(self, child_root, root):
        if child_root == root:
            return
        self.parent[child_root] = root
        self.pattern[root] = max(self.pattern[root], self.pattern[child_root])
        self.size[root] += self.size[child_root]
    monkeypatch.setattr(P.UnionFind, "union_into", union_into)
    _fails(TP.test_phase1_absorbs_the_tuple_phase2_its_fields)


def test_mutation_threshold_inclusive_of_the_next_tensor(monkeypatch):
    import oracle.buckets as B
    from tests import test_oracle_buckets as TB
    orig = B.threshold_buckets

    def bad(numels, threshold, elem_bytes=2, align=256):
        return orig(numels, threshold + 256, elem_bytes, align)   # lets one more tensor in
    monkeypatch.setattr(B, "threshold_buckets", bad)
    _fails(lambda: TB.test_threshold_closed_form_equal_sizes())


def test_mutation_groups_never_checked_for_convexity(monkeypatch):
    import oracle.explicit as X
    from tests import test_oracle_explicit as TX
    monkeypatch.setattr(X, "is_convex", lambda st, nodes: True)
    _fails(TX.test_refused_moves)


def test_mutation_last_pattern_wins(monkeypatch):
    import oracle.patterns as PT
    from tests import test_oracle_patterns as TPT
    orig = PT.match
    monkeypatch.setattr(PT, "match", lambda spec, patterns: orig(spec, list(reversed(patterns))))
    _fails(TPT.test_first_pattern_wins)


def test_mutation_allreduce_ignores_the_channel(monkeypatch):
    import oracle.simulate as S
    from tests import test_oracle_simulate as TS
    orig = S.simulate

    def bad(op_time, edges, tensor_producer, tensor_bytes, buckets, c, d, ar_edges=()):
        # every bucket alone on its own channel: reduce them one at a time
        tot, fin, st, fi = 0.0, None, [], []
        for b in buckets:
            t, fin, s1, f1 = orig(op_time, edges, tensor_producer, tensor_bytes, [b], c, d)
            st += s1
            fi += f1
            tot = max(tot, t)
        if not buckets:
            return orig(op_time, edges, tensor_producer, tensor_bytes, buckets, c, d, ar_edges)
        return tot, fin, st, fi
    monkeypatch.setattr(S, "simulate", bad)
    _fails(TS.test_channel_is_used_in_production_order)


def _patch_op(monkeypatch, op_name, fn):
    orig = E.apply_op
    monkeypatch.setattr(E, "apply_op", lambda op, args, attrs: fn(orig, args, attrs) if op == op_name
                        else orig(op, args, attrs))


def test_mutation_reshape_column_major(monkeypatch):
    _patch_op(monkeypatch, "reshape", lambda orig, args, attrs: np.ascontiguousarray(
        np.asarray(args[0]).reshape(int(attrs[0]), int(attrs[1]), order="F")))
    _fails(TC.test_every_operator_composed)


def test_mutation_transpose_as_reshape(monkeypatch):
    _patch_op(monkeypatch, "transpose", lambda orig, args, attrs: np.ascontiguousarray(
        np.asarray(args[0]).reshape(args[0].shape[::-1])))
    _fails(lambda: TC.test_random_dag_composition(0))


def test_mutation_operands_reversed(monkeypatch):
    _patch_op(monkeypatch, "sub", lambda orig, args, attrs: orig("sub", list(reversed(args)), attrs))
    _fails(TC.test_every_operator_composed)
