"""GB300-native DeepEP-style MoE dispatch / combine.

The product is libep.so (C ABI in include/ep.h, CUDA kernels for sm_103a in
csrc/); `ep` is its thin ctypes binding and `synth` the seeded workload
generator used by tests and the benchmark.
"""
from . import ep, synth  # noqa: F401

__all__ = ["ep", "synth"]
