"""B300-native forward pass of a sparse top-k Mixture-of-Experts layer.

The compute path is hand-written CUDA for sm_103a behind a C ABI
(include/moe.h, built into libmoe_b300.so in this directory).  `binding`
marshals torch tensors into those calls; `workloads` draws the seeded
synthetic inputs.  Importing the package does not load the CUDA library: the
first call through `binding` does, and fails loudly if it is missing.
"""
__all__ = ["binding", "workloads"]
