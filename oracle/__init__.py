"""CPU float64 oracle of the QMoE layer forward (test infrastructure only).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this package; the CUDA library never does.
"""
