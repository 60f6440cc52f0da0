"""CPU oracle for the local Muon step and the alpha-Balanced partition planner.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the ``zero_sharded_gb300``
package, its CUDA library or its C-ABI) may import, call or link anything here;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  The oracle shares no code with the GPU path: it is written
from the Canzona pages ("Canzona: A Unified, Asynchronous, and Load-Balanced
Framework for Distributed Matrix-based Optimizers", arXiv 2602.06079) in plain
Python integers/IEEE doubles (planner) and fp64 NumPy (Muon step).

Modules
-------
planner  -- bucket formation, Eq. 1 start-index split, Algorithm 1
            (alpha-Balanced Greedy LPT), and the objectives J_DP, J_Comm, R_LB.
muon     -- the per-tensor Muon update: momentum (Nesterov), Frobenius
            normalisation, K-step Newton-Schulz, shape scale, apply.

Every function here is pinned by a ``-m "not gpu"`` test against values fixed
by the pages or by mathematics (worked examples, closed forms, invariants);
none is "parity unpinned".
"""
