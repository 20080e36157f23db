"""GB300-native fused causal attention: forward, backward and LSE merge.

The compute path is the C-ABI library ``libattn.so`` (hand-written sm_103a
CUDA kernels) declared in ``include/attn.h``; ``bwd_tcgen05_tmem_gb300.attn``
is a thin ctypes binding over it.  Importing this package loads nothing: the
library is loaded on first use and a missing library raises at that point.
"""
__all__ = ["attn", "synth", "cp"]
