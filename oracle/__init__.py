"""CPU oracle for fused operator-group execution and tensor-fusion packing.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` call it.  It shares no code, table
or constant with the CUDA library; the only module both sides use is
``workloads`` (seeded input generators, no arithmetic of the method).

It is deliberately plain and slow: every operator runs on its own, in
float64, and rounds its result to float32; the pattern-kind table, the
post-dominator tree, the fusion rules and the pack layout are each written
out from the passages they cite:

* ``kinds``     -- OpPatternKind values and the operator table
                   (TVM "Operator Fusion", Operator Pattern Classification).
* ``postdom``   -- immediate post-dominators by LCA on the DAG and the path
                   pattern (TVM, FuseOps > Algorithm, steps 1-2).
* ``partition`` -- CheckPath / CommitFuse with union-find, phases 0, 1 and 2,
                   and the constraints (TVM, FuseOps > Algorithm step 3,
                   Fusion rules).
* ``execute``   -- unfused op-by-op execution (the semantics fusion must keep:
                   DisCo, Introduction, on what op fusion changes).
* ``pack``      -- tensor-fusion layout, bf16 round-to-nearest-even, pack and
                   unpack (DisCo, Introduction, on tensor fusion).
* ``buckets``   -- AllReduce buckets: threshold fusion (DisCo, Related Work,
                   on Horovod and XLA) and neighbour combination (DisCo,
                   Strategy Maker, method (iii)).
* ``explicit``  -- explicit fusion moves: non-duplicate and duplicate fusion
                   of an operator with a predecessor (DisCo, Introduction).
* ``patterns``  -- pattern-based grouping: priority-ordered operator chains
                   with a private-intermediate check (TVM, FuseOpsByPattern).
* ``simulate``  -- the training-step simulator: ready queue, in-order
                   AllReduce channel, linear AllReduce time (DisCo,
                   Simulator and Profiler).

Parity status: every function here is pinned by tests under ``tests/``
(``-m "not gpu"``) against brute force, closed forms, worked examples from the
pages or library routines.  The composition of operators in ``execute`` is
pinned against an independent element-by-element evaluator on small random
DAGs; the full-size chains rely on that composition and the per-operator pins.
"""
from . import kinds, postdom, partition, execute, pack, buckets, explicit, patterns, simulate  # noqa: F401
