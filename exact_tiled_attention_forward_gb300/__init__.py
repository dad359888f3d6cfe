"""Exact tiled attention forward (FlashAttention forward) for GB300 / sm_103a.

The compute path is the C-ABI library ``libfa`` (hand-written CUDA kernels);
this package holds its Python binding and the seeded input generator.
"""
