"""CPU oracle for the deterministic attention backward pass and its tile schedules.

TEST INFRASTRUCTURE ONLY.  This package may be imported by ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``; nothing on the product path (the CUDA library and its
Python binding) imports it, and it imports nothing from the product.

Contents
--------
``attention``
    Plain fp64 softmax-attention forward (O, LSE) and backward (dQ, dK, dV,
    delta), written out from the textbook definition that the DASH pages
    assume ("DASH: Deterministic Attention Scheduling for High-Throughput",
    gist.science technical summary, section 1: the dQ gradient is a sum over
    KV tiles whose order must be fixed).
``dagsim``
    The DAG model of the deterministic backward (compute nodes of cost c,
    reduce nodes of cost r, chain edges, accumulation-order edges; the
    objective is the critical path), the schedules (descending Q-tile
    iteration, shift, symmetric shift, serialized ascending, unordered
    atomics), a longest-path / deadlock evaluator and the zero-weight-edge
    lemma checker (same summary, sections 2.1 and 2.2).

Every function is pinned by tests in ``tests/test_oracle_*.py`` against
finite differences, closed forms, special cases, a library autograd routine
and brute force; the one statement the pages make that is false as printed
(the lemma's "iff" for the critical-path length) is recorded there with a
counterexample.
"""
