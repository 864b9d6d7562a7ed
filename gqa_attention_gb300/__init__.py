"""Grouped-query fused attention forward for one GB300 (sm_103a).

The compute runs in ``libgqa_attn.so`` (CUDA kernels behind a C ABI declared in
``include/gqa_attn.h``); this package is its thin Python binding.  The library
is loaded on first use and a missing or unbuildable library raises: there is no
CPU fallback.
"""
