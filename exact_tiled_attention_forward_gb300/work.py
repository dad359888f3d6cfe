"""Algorithmic work of one attention forward: the FLOP and byte counts the
throughput and roofline figures are quoted against.

* FLOPs: ``4 N_q N_k d`` per query head (the two matrix products), halved
  for causal ("FlashAttention HBM bytes, one head, 8K", "A strong answer" and
  "What interviewers probe next"). For causal with N_q != N_k the visible
  pairs are counted exactly instead.
* Bytes: Q, K and V read once (K and V once per KV head), O written once,
  plus the FP32 LSE row statistic.
"""
from __future__ import annotations


def visible_pairs(n_q: int, n_k: int, causal: bool) -> int:
    """Number of (query, key) pairs that enter the softmax for one head."""
    if not causal:
        return n_q * n_k
    off = n_k - n_q
    total = 0
    # rows whose visible count is clipped to 0 or n_k contribute 0 or n_k
    for i in range(n_q):
        total += min(n_k, max(0, i + off + 1))
    return total


def flops(B: int, H_q: int, N_q: int, N_k: int, d: int, causal: bool) -> float:
    """``4 d`` FLOPs per visible pair (QK^T and PV), all query heads.

    For causal with N_q == N_k this is ``2 N (N + 1) d`` per head; the pages'
    rounded convention ``2 N^2 d`` differs by ``2 N d`` (0.01% at N = 8192).
    """
    if not causal:
        return 4.0 * B * H_q * N_q * N_k * d
    return 4.0 * B * H_q * visible_pairs(N_q, N_k, True) * d


def flops_pages(B: int, H_q: int, N_q: int, N_k: int, d: int, causal: bool) -> float:
    """The pages' convention: ``4 N_q N_k d`` per head, halved when causal."""
    f = 4.0 * B * H_q * N_q * N_k * d
    return f / 2 if causal else f


def bytes_moved(B: int, H_q: int, H_kv: int, N_q: int, N_k: int, d: int, lse: bool = True) -> int:
    """Compulsory bytes: Q, K, V read once, O written once (BF16), LSE written (FP32)."""
    n = 2 * d * (2 * B * H_q * N_q + 2 * B * H_kv * N_k)
    if lse:
        n += 4 * B * H_q * N_q
    return n
