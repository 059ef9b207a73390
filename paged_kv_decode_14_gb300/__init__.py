"""Paged-KV decode attention for GB300 (sm_103a).

Python binding over the C-ABI library ``libpagedkv.so``: ``append`` writes a
step's new K/V into their cache blocks (bf16 or FP8-e4m3), ``attention``
computes decode / causal-verify attention over the paged cache.
"""
