"""B300-native (sm_103a) blockwise ring attention.

The compute lives in ``libringattn.so`` (hand-written CUDA, C ABI declared in
``include/ring_attn.h``); ``ring_attention_02_b300.api`` marshals torch tensors
into those calls.  The shared library is loaded on first use and its absence
is an error: there is no CPU fallback.
"""
__all__ = ["api", "inputs"]
