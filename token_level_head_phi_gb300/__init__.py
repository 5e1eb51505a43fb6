"""GB300-native token-level multi-head linear attention (MHLA) forward pass.

The compute path is ``libmhla.so`` (hand-written sm_103a CUDA kernels behind a
C ABI, declared in ``include/mhla.h``).  ``token_level_head_phi_gb300.binding``
marshals torch tensors into that ABI; ``workloads`` draws seeded synthetic
inputs.  Importing the package loads nothing: the binding loads the library
on first use and raises if it is missing.
"""

__all__ = ["binding", "workloads", "build"]
