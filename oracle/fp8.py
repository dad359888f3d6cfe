"""FP8 (E4M3) inputs for the attention definition — TEST INFRASTRUCTURE ONLY
(see the package docstring: only tests/, the smoke check and bench.py's CPU leg
may use it).

The pages name FP8 only as the next precision step after FP16 on Hopper-class
hardware ("Flash Attention Mechanics...", "FlashAttention 2 and FlashAttention
3"); they define no FP8 arithmetic. The reading here: an FP8 input is a tensor
of E4M3 codes with one per-tensor factor, standing for the values
``decode(code) * descale``; attention over FP8 inputs is the same definition
(``attention.attention_reference``) applied to those values in FP64.

E4M3, from the format's definition: bit 7 sign; bits 3-6 exponent field E
(bias 7); bits 0-2 mantissa M. E = 0: subnormal, M * 2^-9. E = 1..15: normal,
(1 + M/8) * 2^(E-7), except S.1111.111, which is NaN. No infinities; the
largest finite magnitude is 1.75 * 2^8 = 448.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_reference


def e4m3_to_f64(codes) -> np.ndarray:
    """Exact value of each FP8 E4M3 code (uint8) as float64 (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)
    return np.where(c >> 7 == 1, -mag, mag)


def attention_reference_fp8(q, k, v, descale, causal: bool = False, scale: float | None = None):
    """(O, LSE) in FP64 for E4M3 code tensors q, k, v with per-tensor factors
    ``descale = (s_q, s_k, s_v)``: the definition on ``e4m3_to_f64(x) * s_x``."""
    s_q, s_k, s_v = descale
    return attention_reference(e4m3_to_f64(q) * s_q, e4m3_to_f64(k) * s_k, e4m3_to_f64(v) * s_v,
                               causal=causal, scale=scale)


def p_rounding_weight(p):
    """Largest change, per unit of l, that rounding one probability p (relative
    to its row max, 0 < p <= 1) to E4M3 can make, for any reference max the
    kernel holds: the kernel rounds lam * p with 1 <= lam <= 2^8 and divides by
    lam * l, so the change per unit of l is at most
      2^-4 p       where lam p is normal (>= 2^-6; 3 mantissa bits, half spacing
                   2^-4 relative), which holds whenever p >= 2^-6;
      2^-10        where lam p is subnormal (spacing 2^-9), used for
                   2^-10 <= p < 2^-6;
      p            where lam p may round to zero, used for p < 2^-10.
    """
    p = np.asarray(p, dtype=np.float64)
    return np.where(p >= 2.0 ** -6, 2.0 ** -4 * p, np.where(p >= 2.0 ** -10, 2.0 ** -10, p))


def p_rounding_bound_fp8(q, k, v, descale, causal: bool = False, scale: float | None = None):
    """E[b, h, i, t] = sum_j w(p_ij) |v_jt| / l_i with w = ``p_rounding_weight``
    and p_ij = exp(s_ij - max_j s_ij): the most that rounding every P of row i
    to E4M3 before the P V product can move O[i, t] (FP64, materialised per
    row block like ``attention_reference``; masked keys contribute nothing)."""
    from .attention import _ROW_BLOCK, visible_key_count
    s_q, s_k, s_v = descale
    qf, kf, vf = e4m3_to_f64(q) * s_q, e4m3_to_f64(k) * s_k, np.abs(e4m3_to_f64(v) * s_v)
    B, H_q, n_q, d = qf.shape
    H_kv, n_k = kf.shape[1], kf.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    g = H_q // H_kv
    out = np.zeros((B, H_q, n_q, d))
    for b in range(B):
        for h in range(H_q):
            kh, vh = kf[b, h // g], vf[b, h // g]
            for r0 in range(0, n_q, _ROW_BLOCK):
                rows = np.arange(r0, min(n_q, r0 + _ROW_BLOCK))
                s = scale * (qf[b, h, rows] @ kh.T)
                if causal:
                    vis = visible_key_count(rows, n_q, n_k, True)
                    s = np.where(np.arange(n_k)[None, :] < vis[:, None], s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                live = np.isfinite(m)
                p = np.exp(s - np.where(live, m, 0.0))
                l = p.sum(axis=1, keepdims=True)
                w = p_rounding_weight(p)
                out[b, h, rows] = np.where(live, (w @ vh) / np.where(l > 0, l, 1.0), 0.0)
    return out
