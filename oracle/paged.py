"""Decode over a paged K/V cache, FP64 — TEST INFRASTRUCTURE ONLY (see the
package docstring: only tests/, the smoke check and bench.py's CPU leg may use
it).

The pages describe decode as one query against many cached keys ("FlashAttention
HBM bytes, one head, 8K", "What interviewers probe next") and fix no cache
layout. Attention over a paged cache is therefore the same definition,
``attention.attention_reference``, applied to each sequence's keys read out of
its pages in order: key j of sequence b is row ``j mod 128`` of page
``block_table[b][j div 128]`` (every KV head of that page). A sequence with no
key gives O = 0 and LSE = -inf for its rows, the definition's convention for a
row that sees no key. Pinned in tests/test_oracle_paged.py against caches the
test scatters itself from contiguous keys.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_reference

PAGE_KEYS = 128


def gather_sequence(cache, block_table, b: int, n: int) -> np.ndarray:
    """Keys (or values) 0 .. n-1 of sequence b as ``[H_kv][n][d]``, from a
    ``[num_pages][H_kv][128][d]`` cache."""
    j = np.arange(n)
    pages = np.asarray(block_table)[b, j // PAGE_KEYS]
    rows = cache[pages, :, j % PAGE_KEYS]          # [n][H_kv][d]
    return np.ascontiguousarray(np.transpose(rows, (1, 0, 2)))


def paged_attention_reference(q, k_cache, v_cache, block_table, seqlens, causal: bool = False,
                              scale: float | None = None):
    """(O, LSE) in FP64 for q ``[B][H_q][N_q][d]`` against each sequence's
    ``seqlens[b]`` keys (0 <= seqlens[b] <= 128 * block_table.shape[1])."""
    B, H_q, n_q, d = q.shape
    o = np.zeros((B, H_q, n_q, d), dtype=np.float64)
    lse = np.full((B, H_q, n_q), -np.inf, dtype=np.float64)
    for b in range(B):
        n = int(seqlens[b])
        assert 0 <= n <= PAGE_KEYS * np.asarray(block_table).shape[1]
        if n == 0:
            continue
        kb = gather_sequence(k_cache, block_table, b, n)[None]
        vb = gather_sequence(v_cache, block_table, b, n)[None]
        ob, lb = attention_reference(q[b:b + 1], kb, vb, causal=causal, scale=scale)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse
