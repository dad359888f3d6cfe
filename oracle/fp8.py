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
