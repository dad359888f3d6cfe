"""FP64 oracle of the exact attention forward (test infrastructure only).

Sources (by page and section):

* "Why is standard attention memory-bound, and how does FlashAttention fix
  it?" (interview.clozo.ai), Step 1: scaled dot-product attention is the
  softmax of the scaled product of Q and K^T, multiplied by V.
* "Flash Attention Mechanics: How Tiled Attention Fits in SRAM"
  (interviewprepkit.dev), section "Why Standard Attention Is Memory-Bound"
  (softmax(QK^T / sqrt(d)) V) and section "The Tiling Algorithm" (the
  standard attention routine: full score matrix per head, subtract the row
  max, exponentiate, normalise, multiply by V; the tiled routine with the
  running max / running sum / unnormalised output update).
* Same page 3, Step 3 and "Follow-up questions": the online softmax keeps a
  running max and running sum and rescales the sum and partial output by
  exp(m_old - m_new) when the max rises; the final output is divided by the
  final sum.

Readings where the pages are silent (the plainest reading each time):

* LSE (the per-row statistic kept for the backward pass, page 3 Step 4) is
  the natural-log log-sum-exp of the *scaled* scores: ``m + ln(l)``.
* Causal with N_q != N_k: bottom-right alignment, query i sees key j iff
  ``j <= i + (N_k - N_q)``. A row with no visible key has O = 0, LSE = -inf.
* GQA: query head h reads KV head ``h // (H_q // H_kv)``.
* Inputs are BF16 bit patterns, widened exactly to FP64 before any
  arithmetic; ``scale`` is used exactly as given.
"""
from __future__ import annotations

import math

import numpy as np

_ROW_BLOCK = 512  # rows of S materialised at a time (bounds memory, not arithmetic)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)


def to_f64(x: np.ndarray) -> np.ndarray:
    """Exact widening of an input tensor to float64: floating-point arrays
    (binary16, 32, 64) by value, 16-bit integer arrays as bfloat16 bit patterns."""
    x = np.asarray(x)
    if np.issubdtype(x.dtype, np.floating):
        return x.astype(np.float64)
    return bf16_to_f64(x)


def visible_key_count(i: np.ndarray | int, n_q: int, n_k: int, causal: bool):
    """Number of keys query row ``i`` may attend to (keys 0 .. count-1).

    Non-causal: all ``n_k``. Causal, bottom-right aligned (the reading above):
    ``clip(i + n_k - n_q + 1, 0, n_k)``. For n_q == n_k this is the
    lower-triangular mask of page 1, "What interviewers probe next".
    """
    if not causal:
        return np.full(np.shape(i), n_k) if np.ndim(i) else n_k
    return np.clip(np.asarray(i) + (n_k - n_q) + 1, 0, n_k)


def _softmax_rows(s: np.ndarray):
    """Row softmax with the row max subtracted (page 2, "The Tiling Algorithm",
    standard attention routine). ``s`` may hold -inf for masked entries.

    Returns (P, m, l) with P = exp(s - m) / l, m = row max, l = row sum of
    exp(s - m). Rows that are entirely -inf give P = 0, m = -inf, l = 0.
    """
    m = s.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe)
    l = e.sum(axis=-1, keepdims=True)
    p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
    return p, m, l


def _head_rows(qh, kh, vh, rows, n_q, n_k, causal, scale):
    """O and LSE for the listed query rows of one head, S materialised."""
    s = scale * (qh[rows] @ kh.T)                       # scores, FP64
    if causal:
        vis = visible_key_count(rows, n_q, n_k, True)
        cols = np.arange(n_k)
        s = np.where(cols[None, :] < vis[:, None], s, -np.inf)
    p, m, l = _softmax_rows(s)
    o = p @ vh
    with np.errstate(divide="ignore"):
        lse = np.where(l[:, 0] > 0, m[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)),
                       -np.inf)
    return o, lse


def attention_reference(q, k, v, causal: bool = False, scale: float | None = None):
    """The definition, materialised: for every (batch, query head),
    ``S = scale * Q K^T``, mask, ``P = softmax_row(S)``, ``O = P V`` and
    ``LSE = m + ln l``.

    ``q``: bf16 bits (or float16 values) ``[B][H_q][N_q][d]``; ``k``, ``v``: ``[B][H_kv][N_k][d]``.
    Returns ``(O, LSE)`` as float64 arrays ``[B][H_q][N_q][d]``, ``[B][H_q][N_q]``.
    """
    B, H_q, n_q, d = q.shape
    _, H_kv, n_k, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = H_q // H_kv
    o = np.zeros((B, H_q, n_q, d))
    lse = np.zeros((B, H_q, n_q))
    for b in range(B):
        for hk in range(H_kv):
            kh = to_f64(k[b, hk])
            vh = to_f64(v[b, hk])
            for h in range(hk * g, (hk + 1) * g):
                qh = to_f64(q[b, h])
                for r0 in range(0, n_q, _ROW_BLOCK):
                    rows = np.arange(r0, min(n_q, r0 + _ROW_BLOCK))
                    o[b, h, rows], lse[b, h, rows] = _head_rows(qh, kh, vh, rows, n_q, n_k,
                                                                causal, scale)
    return o, lse


def attention_rows(q, k, v, b: int, h: int, rows, causal: bool = False,
                   scale: float | None = None):
    """Same definition for a chosen set of query rows of one (batch, head).

    Each row of the result depends only on its own query row and on K, V,
    so a sample of rows is checked exactly at any problem size.
    """
    _, H_q, n_q, d = q.shape
    _, H_kv, n_k, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    hk = h // (H_q // H_kv)
    rows = np.asarray(rows, dtype=np.int64)
    qh = to_f64(q[b, h, rows])
    kh = to_f64(k[b, hk])
    vh = to_f64(v[b, hk])
    o = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    for r0 in range(0, len(rows), _ROW_BLOCK):
        sl = slice(r0, r0 + _ROW_BLOCK)
        # rows are re-indexed into the gathered qh block; the mask uses the true row index
        s = scale * (qh[sl] @ kh.T)
        if causal:
            vis = visible_key_count(rows[sl], n_q, n_k, True)
            s = np.where(np.arange(n_k)[None, :] < vis[:, None], s, -np.inf)
        p, m, l = _softmax_rows(s)
        o[sl] = p @ vh
        with np.errstate(divide="ignore"):
            lse[sl] = np.where(l[:, 0] > 0,
                               m[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    return o, lse


def online_softmax_blocks(score_blocks, value_blocks=None):
    """Streaming softmax over a row split into blocks (page 3, Step 3 and
    "What is online softmax?"; page 2, "The Tiling Algorithm").

    Keeps a running max ``m`` and running sum ``l``; when a block raises the
    max from m_old to m_new, the running sum and the partial output are
    multiplied by exp(m_old - m_new) before the block's own terms are added.
    ``score_blocks`` is a list of 1-D score arrays of one row; ``value_blocks``
    (optional) the matching ``[len(block), d]`` value rows. Returns
    ``(m, l, o)`` with ``o`` the unnormalised weighted sum (None if no values).
    """
    m = -np.inf
    l = 0.0
    o = None
    for i, s in enumerate(score_blocks):
        s = np.asarray(s, dtype=np.float64)
        m_new = max(m, float(s.max())) if s.size else m
        if m_new == -np.inf:
            continue
        alpha = math.exp(m - m_new) if m != -np.inf else 0.0
        e = np.exp(s - m_new)
        l = alpha * l + float(e.sum())
        if value_blocks is not None:
            contrib = e @ np.asarray(value_blocks[i], dtype=np.float64)
            o = contrib if o is None else alpha * o + contrib
        m = m_new
    return m, l, o


def attention_tiled_online(q, k, v, block_q: int, block_k: int, causal: bool = False,
                           scale: float | None = None):
    """Tiled restatement used as a self-check of ``attention_reference``:
    query blocks outermost, K/V blocks inner, online softmax state (m, l, o)
    per query row, divide by l once at the end (page 2, "The Tiling
    Algorithm"). FP64 throughout; ragged last blocks via ``min``.
    Same argument and return conventions as ``attention_reference``.
    """
    B, H_q, n_q, d = q.shape
    _, H_kv, n_k, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = H_q // H_kv
    out = np.zeros((B, H_q, n_q, d))
    lse = np.zeros((B, H_q, n_q))
    for b in range(B):
        for h in range(H_q):
            qh = to_f64(q[b, h])
            kh = to_f64(k[b, h // g])
            vh = to_f64(v[b, h // g])
            for q0 in range(0, n_q, block_q):
                q1 = min(q0 + block_q, n_q)
                rows = np.arange(q0, q1)
                m = np.full((q1 - q0, 1), -np.inf)
                l = np.zeros((q1 - q0, 1))
                o = np.zeros((q1 - q0, d))
                for k0 in range(0, n_k, block_k):
                    k1 = min(k0 + block_k, n_k)
                    s = scale * (qh[q0:q1] @ kh[k0:k1].T)
                    if causal:
                        vis = visible_key_count(rows, n_q, n_k, True)
                        s = np.where(np.arange(k0, k1)[None, :] < vis[:, None], s, -np.inf)
                    m_blk = s.max(axis=1, keepdims=True)
                    m_new = np.maximum(m, m_blk)
                    ref = np.where(np.isfinite(m_new), m_new, 0.0)
                    alpha = np.exp(m - ref)        # exp(-inf) = 0 on the first live block
                    e = np.exp(s - ref)
                    l = alpha * l + e.sum(axis=1, keepdims=True)
                    o = alpha * o + e @ vh[k0:k1]
                    m = m_new
                live = l[:, 0] > 0
                out[b, h, q0:q1] = np.where(live[:, None], o / np.where(l > 0, l, 1.0), 0.0)
                with np.errstate(divide="ignore"):
                    lse[b, h, q0:q1] = np.where(
                        live, m[:, 0] + np.log(np.where(live, l[:, 0], 1.0)), -np.inf)
    return out, lse


def brute_force_attention(q, k, v, causal: bool = False, scale: float | None = None):
    """Pure-Python triple loop with no max subtraction, for tiny shapes only:
    o_i = sum_j exp(s_ij) v_j / sum_j exp(s_ij), lse_i = ln sum_j exp(s_ij).
    Inputs are nested lists / arrays of floats shaped like the BF16 tensors
    (already widened); returns nested lists.
    """
    B, H_q, n_q, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    H_kv, n_k = len(k[0]), len(k[0][0])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = H_q // H_kv
    O = [[[[0.0] * d for _ in range(n_q)] for _ in range(H_q)] for _ in range(B)]
    L = [[[0.0] * n_q for _ in range(H_q)] for _ in range(B)]
    for b in range(B):
        for h in range(H_q):
            for i in range(n_q):
                num = [0.0] * d
                den = 0.0
                for j in range(n_k):
                    if causal and j > i + (n_k - n_q):
                        continue
                    s = 0.0
                    for t in range(d):
                        s += float(q[b][h][i][t]) * float(k[b][h // g][j][t])
                    w = math.exp(scale * s)
                    den += w
                    for t in range(d):
                        num[t] += w * float(v[b][h // g][j][t])
                O[b][h][i] = [x / den for x in num] if den > 0 else [0.0] * d
                L[b][h][i] = math.log(den) if den > 0 else -math.inf
    return O, L


def merge_partials(ms, ls, os_):
    """Combine softmax partials of disjoint key ranges of the same rows
    (the online-softmax merge of page 2, "The Tiling Algorithm", applied to
    whole ranges; page 3, "Does FlashAttention help when generating one token
    at a time?" splits the key sequence across thread blocks and combines).

    ``ms``, ``ls``: lists of ``[rows]`` arrays (max and sum of exp(s - m) of
    each range); ``os_``: list of ``[rows, d]`` unnormalised outputs.
    Returns the normalised ``(O, LSE)``; rows with no live range give 0, -inf.
    """
    ms = [np.asarray(x, dtype=np.float64) for x in ms]
    m = np.max(np.stack(ms), axis=0)
    ref = np.where(np.isfinite(m), m, 0.0)
    l = np.zeros_like(m)
    o = np.zeros_like(np.asarray(os_[0], dtype=np.float64))
    for mi, li, oi in zip(ms, ls, os_):
        w = np.where(np.isfinite(mi), np.exp(np.where(np.isfinite(mi), mi, 0.0) - ref), 0.0)
        l = l + w * np.asarray(li, dtype=np.float64)
        o = o + w[:, None] * np.asarray(oi, dtype=np.float64)
    live = l > 0
    out = np.where(live[:, None], o / np.where(live, l, 1.0)[:, None], 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(live, ref + np.log(np.where(live, l, 1.0)), -np.inf)
    return out, lse
