"""GB300-native (sm_103a) MoE routing, dispatch and fused grouped GEMM.

The compute path lives in the CUDA shared library built from ``csrc/``; the
Python module ``binding`` only marshals arguments into its C ABI (see
``include/moe.h``).  ``workloads`` draws the seeded synthetic inputs.
"""
__all__ = ["binding", "workloads"]
