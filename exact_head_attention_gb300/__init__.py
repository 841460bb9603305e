"""exact_head_attention_gb300: exact fused multi-head attention (forward and
backward) for GB300 (sm_103a), exposed as a C-ABI shared library
(``include/exattn.h``) with a thin ctypes binding (``exattn``).

Importing the package does not load the CUDA library; ``exattn`` loads it on
first use and raises if it is missing.
"""
__all__ = ["workloads", "exattn"]
