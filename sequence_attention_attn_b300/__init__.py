"""B300-native DiT blockwise attention: tcgen05/TMEM/TMA attention forward with
on-chip chunk merging, a standalone log-sum-exp merge and the classifier-free
guidance combine, behind the C ABI of ``libditattn.so``.

Importing the package loads nothing; the CUDA library is loaded by the first
call into :mod:`sequence_attention_attn_b300.dit_attn`, which raises if the
library is missing (there is no CPU fallback).
"""
__all__ = ["dit_attn", "workloads"]
