"""GB300 (sm_103a) hybrid prefill+decode attention.

The compute path is the C-ABI library ``libpod_attn.so`` (CUDA kernels for sm_103a) declared
in ``include/pod_attn.h``; ``hybrid_prefill_decode_gb300.binding`` marshals arguments to it.
Importing this package loads nothing: the library is loaded on first use of the binding, and
fails loudly if it has not been built.
"""
__all__ = ["binding", "workloads", "roofline"]
