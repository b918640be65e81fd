"""GB300-native batched tree speculative-sampling verify (EAGLE / SpecInfer style).

The compute path is the C-ABI library built from ``csrc/`` (CUDA for sm_103a);
``binding`` marshals torch tensors into it.  Importing this package does not load
the library; the first call into ``binding`` does, and raises if it is missing.
"""

__all__ = ["binding", "workloads"]
