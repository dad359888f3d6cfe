"""FP64 gradients of exact attention — TEST INFRASTRUCTURE ONLY (see the package
docstring: only tests/, the smoke check and bench.py's CPU leg may use it).

What the pages fix: the backward pass recomputes the scores tile by tile from
Q, K and the small per-row statistics saved by the forward instead of storing
the N x N matrices ("Why is standard attention memory-bound...", Step 4 and
"Why does the backward pass recompute the scores?"). They print no gradient
formulas, so this module writes out the derivative of the definition
O = softmax(scale Q K^T) V (with the forward's mask and GQA mapping) by the
chain rule, materialising S and P head by head:

    dV = P^T dO                 dP = dO V^T
    D_i = sum_t dO_it O_it      (= sum_j P_ij dP_ij)
    dS = P * (dP - D)           (the softmax Jacobian applied row by row)
    dQ = scale dS K             dK = scale dS^T Q

dK and dV of a KV head sum the contributions of every query head that reads
it. A row that sees no key has P = 0 and contributes nothing. These formulas
are pinned in tests/test_oracle_backward.py against central finite
differences of the forward oracle, not against themselves.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import to_f64, visible_key_count


def _probabilities(qh, kh, n_q, n_k, causal, scale):
    """P (rows x keys) of one head, FP64, masked rows all zero."""
    s = scale * (qh @ kh.T)
    if causal:
        vis = visible_key_count(np.arange(n_q), n_q, n_k, True)
        s = np.where(np.arange(n_k)[None, :] < vis[:, None], s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    live = np.isfinite(m[:, 0])
    e = np.exp(s - np.where(live[:, None], m, 0.0))
    e[~live] = 0.0
    l = e.sum(axis=1, keepdims=True)
    return np.where(live[:, None], e / np.where(l > 0, l, 1.0), 0.0)


def attention_backward(q, k, v, do, causal: bool = False, scale: float | None = None):
    """(dQ, dK, dV) in float64 for upstream gradient dO.

    ``q``, ``do``: ``[B][H_q][N_q][d]``; ``k``, ``v``: ``[B][H_kv][N_k][d]``;
    bfloat16 bit patterns, binary16 or float64 arrays (widened exactly)."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    B, H_q, n_q, d = q.shape
    H_kv, n_k = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = H_q // H_kv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H_q):
            hk = h // g
            qh, kh, vh, doh = q[b, h], k[b, hk], v[b, hk], do[b, h]
            p = _probabilities(qh, kh, n_q, n_k, causal, scale)
            o = p @ vh
            dv[b, hk] += p.T @ doh
            dp = doh @ vh.T
            dd = (doh * o).sum(axis=1, keepdims=True)
            ds = p * (dp - dd)
            dq[b, h] = scale * (ds @ kh)
            dk[b, hk] += scale * (ds.T @ qh)
    return dq, dk, dv


def forward_loss(q, k, v, do, causal: bool = False, scale: float | None = None) -> float:
    """sum(dO * O) in FP64: the scalar whose gradient attention_backward returns
    (used by the finite-difference pins)."""
    from .attention import attention_reference
    o, _ = attention_reference(q, k, v, causal=causal, scale=scale)
    return float((to_f64(do) * o).sum())


def backward_error_terms(q, k, v, do, causal: bool = False, scale: float | None = None,
                         parts: bool = False):
    """Magnitudes that bound what rounding the method's own precision does to
    each gradient (for the tolerance of a 16-bit backward; FP64, same shapes as
    attention_backward's results):

    * dQ: scale |dS| |K|  +  scale Dabs * (P |K|), with Dabs_i = sum_t |dO_it O_it|
      (dS is rounded before the dS K product; O enters D rounded to 16 bits);
    * dK: scale |dS|^T |Q|  +  scale P^T (Dabs * |Q|);
    * dV: P^T |dO| (P is rounded before the P^T dO product).
    A gradient computed with unit roundoff u is within about u (terms + |gradient|).
    With ``parts`` the terms come back one by one, as a dict: ``dq_ds``, ``dq_d``,
    ``dk_ds``, ``dk_d``, ``dv_p`` (the first-order effect of rounding dS, D's O,
    and P respectively)."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    B, H_q, n_q, d = q.shape
    H_kv, n_k = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = H_q // H_kv
    out = {"dq_ds": np.zeros_like(q), "dq_d": np.zeros_like(q), "dk_ds": np.zeros_like(k),
           "dk_d": np.zeros_like(k), "dv_p": np.zeros_like(v)}
    for b in range(B):
        for h in range(H_q):
            hk = h // g
            qh, kh, vh, doh = q[b, h], k[b, hk], v[b, hk], do[b, h]
            p = _probabilities(qh, kh, n_q, n_k, causal, scale)
            o = p @ vh
            dp = doh @ vh.T
            ds = p * (dp - (doh * o).sum(axis=1, keepdims=True))
            dabs = np.abs(doh * o).sum(axis=1, keepdims=True)
            out["dq_ds"][b, h] = scale * (np.abs(ds) @ np.abs(kh))
            out["dq_d"][b, h] = scale * (dabs * (p @ np.abs(kh)))
            out["dk_ds"][b, hk] += scale * (np.abs(ds).T @ np.abs(qh))
            out["dk_d"][b, hk] += scale * (p.T @ (dabs * np.abs(qh)))
            out["dv_p"][b, hk] += p.T @ np.abs(doh)
    if parts:
        return out
    return out["dq_ds"] + out["dq_d"], out["dk_ds"] + out["dk_d"], out["dv_p"]
