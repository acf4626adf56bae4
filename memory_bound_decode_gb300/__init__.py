"""GB300-native decode GEMV: y = W·x with BF16 weights, FP32 accumulation.

The compute path is the C-ABI library ``libgemv.so`` built from ``csrc/``;
``binding`` marshals arguments to it. Importing this package loads nothing:
the library is loaded on first use and a missing library is an error, never a
fallback.
"""
__all__ = ["binding", "inputs", "roofline", "workloads"]
