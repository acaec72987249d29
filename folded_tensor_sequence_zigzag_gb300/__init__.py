"""GB300-native TSP-folded transformer block (zigzag causal partitioning).

The compute lives in libtsp.so (CUDA, sm_103a) behind the C ABI declared in
include/tsp.h; ``folded_tensor_sequence_zigzag_gb300.tsp`` is its ctypes
binding.  Importing the package does not load the library: the first call
through the binding does, and raises if it is missing.
"""
__all__ = ["tsp", "inputs", "build"]
