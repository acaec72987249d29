"""CPU float64 oracle for the TSP-folded block (test infrastructure only).

Imported only by tests/, the smoke check and the benchmark's CPU-baseline
leg.  The library itself never imports it.
"""
from .tsp_oracle import *  # noqa: F401,F403
