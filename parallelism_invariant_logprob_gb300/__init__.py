"""Batch- and parallelism-invariant bf16 GEMM, RMSNorm, MoE expert layer and
selected-token logprob for NVIDIA GB300 (sm_103a).

The compute path is the CUDA library ``libiso.so`` (hand-written tcgen05 /
TMA kernels behind a C ABI declared in ``include/iso.h``).  ``binding`` is a
thin ctypes layer over it; importing this package does not load the library.
"""
__all__ = ["binding", "inputs"]
