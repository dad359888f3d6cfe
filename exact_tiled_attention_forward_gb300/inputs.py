"""Seeded synthetic inputs for the attention forward: BF16 (or FP16) Q, K, V ~ N(0, 1).

This module is the only code shared by the CUDA path's callers (tests, bench)
and the FP64 oracle. It holds no attention arithmetic: it only draws numbers.

Recipe (fixed, so a seed names one input on every machine that runs it):

* counter-based generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014; finaliser constants as
  published by Vigna). Element ``i`` of stream ``s`` under seed ``seed`` is the
  finaliser applied to ``key(seed, s) + (i + 1) * GAMMA``.
* normal deviates: Box-Muller on pairs of 53-bit uniforms, in float64.
* storage: float64 -> float32 (round to nearest even) -> bfloat16 (round to
  nearest even), kept as raw ``uint16`` bit patterns; or, for FP16 inputs,
  float64 -> IEEE binary16 (round to nearest even, numpy's conversion), kept as
  ``numpy.float16`` arrays. The array's dtype tells the two apart.
* "1% of K rows scaled by 8": for each (batch, kv-head), ``round(0.01 * N_k)``
  rows are picked without replacement (the rows with the smallest draws of a
  separate stream) and multiplied by 8, which is exact in bfloat16 and in
  binary16 (at these magnitudes).

Layouts: Q is ``[B][H_q][N_q][d]``, K and V are ``[B][H_kv][N_k][d]``, all
contiguous row-major.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_Q, STREAM_K, STREAM_V, STREAM_ROWS, STREAM_DO, STREAM_PAGES = 1, 2, 3, 4, 5, 6

_CHUNK = 1 << 22  # elements generated per numpy pass (bounds temporaries)


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    x = np.array([(seed * 0x100000001B3 + stream * 0x632BE59BD9B4E019) & (2**64 - 1)],
                 dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(x + GAMMA)[0]


def uniform_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit draws ``start .. start+count-1`` of one stream."""
    key = _stream_key(seed, stream)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * GAMMA)


def normal_f64(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` standard normal deviates (Box-Muller), float64."""
    return _normal_slice(seed, stream, 0, count)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 (RNE); returns uint16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f64_to_f16(x: np.ndarray) -> np.ndarray:
    """float64 -> IEEE binary16, round to nearest even (numpy's conversion)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)


E4M3_MAX = 448.0   # largest finite FP8 E4M3 value (1.75 * 2^8)


def f64_to_e4m3(x: np.ndarray) -> np.ndarray:
    """float64 -> FP8 E4M3 codes (uint8): 1 sign bit, 4 exponent bits with bias
    7, 3 mantissa bits, subnormals below 2^-6, no infinities (S.1111.111 is NaN).
    Round to nearest, ties to even, saturating to +-448 (as a "satfinite"
    conversion does); NaN maps to 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
    a = np.minimum(np.abs(np.nan_to_num(x, nan=0.0)), E4M3_MAX)
    _, ex = np.frexp(a)                         # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)                  # unbiased exponent; subnormals share 2^-6's
    q = np.rint(np.ldexp(a, 3 - e))             # significand in eighths, ties to even
    carry = q >= 16                             # rounded up to the next binade
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q)
    normal = q >= 8
    code = np.where(normal, ((e + 7) << 3) + (q - 8), q).astype(np.uint8)
    code = code | sign
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def e4m3_power_of_two_scale(x: np.ndarray) -> float:
    """The smallest power of two s with max|x| / s <= 448 (a per-tensor scale
    that keeps every value in range; 1.0 for an all-zero tensor)."""
    amax = float(np.max(np.abs(x))) if np.size(x) else 0.0
    if amax == 0.0:
        return 1.0
    return float(2.0 ** math.ceil(math.log2(amax / E4M3_MAX)))


def normal_f16(seed: int, stream: int, shape) -> np.ndarray:
    """The deviates of ``normal_bf16``'s stream, rounded to binary16 instead."""
    count = int(np.prod(shape))
    out = np.empty(count, dtype=np.float16)
    for lo in range(0, count, 2 * _CHUNK):
        hi = min(count, lo + 2 * _CHUNK)
        out[lo:hi] = f64_to_f16(_normal_slice(seed, stream, lo, hi))
    return out.reshape(shape)


def normal_bf16(seed: int, stream: int, shape) -> np.ndarray:
    count = int(np.prod(shape))
    out = np.empty(count, dtype=np.uint16)
    for lo in range(0, count, 2 * _CHUNK):
        hi = min(count, lo + 2 * _CHUNK)
        # draw the whole stream prefix-consistently: element i always uses pair i//2
        z = _normal_slice(seed, stream, lo, hi)
        out[lo:hi] = f64_to_bf16_bits(z)
    return out.reshape(shape)


def _normal_slice(seed: int, stream: int, lo: int, hi: int) -> np.ndarray:
    """Normal deviates for elements [lo, hi) of a stream (lo even)."""
    assert lo % 2 == 0
    p0, p1 = lo // 2, (hi + 1) // 2
    r = uniform_u64(seed, stream, 2 * p0, 2 * (p1 - p0))
    a = (r[0::2] >> np.uint64(11)).astype(np.float64)
    b = (r[1::2] >> np.uint64(11)).astype(np.float64)
    u1 = (a + 1.0) * (1.0 / 9007199254740992.0)
    u2 = b * (1.0 / 9007199254740992.0)
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * math.pi * u2
    z = np.empty(2 * (p1 - p0), dtype=np.float64)
    z[0::2] = rad * np.cos(ang)
    z[1::2] = rad * np.sin(ang)
    return z[: hi - lo]


def scaled_rows(seed: int, n_bh: int, n_k: int, frac: float) -> np.ndarray:
    """Row indices (per flattened (batch, kv-head)) chosen for the x8 scaling.

    Returns an int64 array of shape ``[n_bh, round(frac * n_k)]``.
    """
    n_pick = int(round(frac * n_k))
    picks = np.empty((n_bh, n_pick), dtype=np.int64)
    for bh in range(n_bh):
        r = uniform_u64(seed, STREAM_ROWS, bh * n_k, n_k)
        picks[bh] = np.sort(np.argsort(r, kind="stable")[:n_pick])
    return picks


@dataclasses.dataclass
class AttentionInputs:
    """One seeded problem. Arrays hold bfloat16 bit patterns (uint16), or
    binary16 values (numpy.float16) when ``dtype`` is "f16"."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    B: int
    H_q: int
    H_kv: int
    N_q: int
    N_k: int
    d: int
    causal: bool
    scale: float
    dtype: str = "bf16"
    # FP8 ("e4m3") inputs only: per-tensor factors (q, k, v) that turn a decoded
    # code back into the value it stands for (x = decode(code) * descale)
    descale: tuple | None = None

    @property
    def shape_args(self):
        return (self.B, self.H_q, self.H_kv, self.N_q, self.N_k, self.d)


def make_inputs(B: int, H_q: int, H_kv: int, N_q: int, N_k: int, d: int, *,
                causal: bool = False, scale: float | None = None, seed: int = 0,
                k_row_frac: float = 0.0, k_row_factor: float = 8.0,
                dtype: str = "bf16") -> AttentionInputs:
    """Draw Q, K, V for one configuration (all ~ N(0, 1); dtype "bf16", "f16",
    or "e4m3": FP8 codes of x / s with s = ``e4m3_power_of_two_scale`` per
    tensor, the deviates taken in FP64 from the same streams)."""
    if dtype == "e4m3":
        return _make_inputs_e4m3(B, H_q, H_kv, N_q, N_k, d, causal=causal, scale=scale, seed=seed,
                                 k_row_frac=k_row_frac, k_row_factor=k_row_factor)
    if dtype not in ("bf16", "f16"):
        raise ValueError(f"dtype must be 'bf16', 'f16' or 'e4m3', not {dtype!r}")
    draw = normal_f16 if dtype == "f16" else normal_bf16
    q = draw(seed, STREAM_Q, (B, H_q, N_q, d))
    k = draw(seed, STREAM_K, (B, H_kv, N_k, d))
    v = draw(seed, STREAM_V, (B, H_kv, N_k, d))
    if k_row_frac > 0.0:
        rows = scaled_rows(seed, B * H_kv, N_k, k_row_frac)
        kf = k.reshape(B * H_kv, N_k, d)
        for bh in range(B * H_kv):
            sel = kf[bh, rows[bh]]
            if dtype == "f16":
                kf[bh, rows[bh]] = f64_to_f16(sel.astype(np.float64) * k_row_factor)
            else:
                kf[bh, rows[bh]] = f64_to_bf16_bits(bf16_bits_to_f32(sel).astype(np.float64) * k_row_factor)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return AttentionInputs(q, k, v, B, H_q, H_kv, N_q, N_k, d, bool(causal), float(scale), dtype)


def _normal_array(seed: int, stream: int, shape) -> np.ndarray:
    count = int(np.prod(shape))
    out = np.empty(count, dtype=np.float64)
    for lo in range(0, count, 2 * _CHUNK):
        hi = min(count, lo + 2 * _CHUNK)
        out[lo:hi] = _normal_slice(seed, stream, lo, hi)
    return out.reshape(shape)


def _make_inputs_e4m3(B, H_q, H_kv, N_q, N_k, d, *, causal, scale, seed, k_row_frac, k_row_factor):
    q = _normal_array(seed, STREAM_Q, (B, H_q, N_q, d))
    k = _normal_array(seed, STREAM_K, (B, H_kv, N_k, d))
    v = _normal_array(seed, STREAM_V, (B, H_kv, N_k, d))
    if k_row_frac > 0.0:
        rows = scaled_rows(seed, B * H_kv, N_k, k_row_frac)
        kf = k.reshape(B * H_kv, N_k, d)
        for bh in range(B * H_kv):
            kf[bh, rows[bh]] *= k_row_factor
    codes, descale = [], []
    for x in (q, k, v):
        s = e4m3_power_of_two_scale(x)
        codes.append(f64_to_e4m3(x / s))
        descale.append(s)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return AttentionInputs(codes[0], codes[1], codes[2], B, H_q, H_kv, N_q, N_k, d, bool(causal), float(scale),
                           "e4m3", tuple(descale))


def grad_output(a: AttentionInputs, seed: int = 0) -> np.ndarray:
    """dO for a backward pass of `a`: N(0, 1) in a's storage type, shaped like O."""
    shape = (a.B, a.H_q, a.N_q, a.d)
    return normal_f16(seed, STREAM_DO, shape) if a.dtype == "f16" else normal_bf16(seed, STREAM_DO, shape)


PAGE_KEYS = 128   # keys per page of a paged K/V cache


@dataclasses.dataclass
class PagedInputs:
    """A decode problem whose K/V cache is paged. ``q`` ``[B][H_q][N_q][d]``;
    ``k_cache``, ``v_cache`` ``[num_pages][H_kv][128][d]``; ``block_table``
    int32 ``[B][max_pages]`` (key j of sequence b is row j % 128 of page
    ``block_table[b][j // 128]``); ``seqlens`` int32 ``[B]``. Element storage
    as in ``AttentionInputs``."""
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_table: np.ndarray
    seqlens: np.ndarray
    B: int
    H_q: int
    H_kv: int
    N_q: int
    d: int
    causal: bool
    scale: float
    dtype: str = "bf16"


def make_paged(B: int, H_q: int, H_kv: int, N_q: int, seqlens, d: int, *, causal: bool = False,
               scale: float | None = None, seed: int = 0, spare_pages: int = 3, max_pages: int | None = None,
               k_row_frac: float = 0.0, dtype: str = "bf16") -> PagedInputs:
    """Q, K, V drawn as ``make_inputs`` draws them (K and V for
    ``max_pages * 128`` keys per sequence), then K/V laid out in pages.

    Sequence b keeps its first ``ceil(seqlens[b] / 128)`` key blocks, each in a
    page of its own; pages are numbered in a seeded random order, with
    ``spare_pages`` extra pages (random data no sequence owns) among them. The
    keys of a sequence's last page past its length keep their drawn values, and
    block-table entries past a sequence's last page hold seeded page numbers:
    neither may change a result. ``max_pages`` defaults to the longest
    sequence's page count."""
    seqlens = np.asarray(seqlens, dtype=np.int64)
    assert seqlens.shape == (B,) and (seqlens >= 0).all()
    used = (seqlens + PAGE_KEYS - 1) // PAGE_KEYS
    if max_pages is None:
        max_pages = max(1, int(used.max()) if B else 1)
    assert (used <= max_pages).all()
    a = make_inputs(B, H_q, H_kv, N_q, max_pages * PAGE_KEYS, d, causal=causal, scale=scale, seed=seed,
                    k_row_frac=k_row_frac, dtype=dtype)
    num_pages = int(used.sum()) + spare_pages
    order = np.argsort(uniform_u64(seed, STREAM_PAGES, 0, max(num_pages, 1)), kind="stable")[:num_pages]
    k_cache = np.empty((num_pages, H_kv, PAGE_KEYS, d), dtype=a.k.dtype)
    v_cache = np.empty_like(k_cache)
    table = (uniform_u64(seed, STREAM_PAGES, num_pages, B * max_pages) % np.uint64(max(num_pages, 1)))
    table = table.astype(np.int32).reshape(B, max_pages)
    slot = 0
    for b in range(B):
        for j in range(int(used[b])):
            page = int(order[slot])
            slot += 1
            table[b, j] = page
            k_cache[page] = a.k[b, :, j * PAGE_KEYS:(j + 1) * PAGE_KEYS]
            v_cache[page] = a.v[b, :, j * PAGE_KEYS:(j + 1) * PAGE_KEYS]
    # the spare pages: data of other seeded draws
    spare = order[slot:]
    if len(spare):
        draw = normal_f16 if dtype == "f16" else normal_bf16
        fill = draw(seed + 1, STREAM_K, (len(spare), H_kv, PAGE_KEYS, d))
        k_cache[spare] = fill
        v_cache[spare] = fill[::-1]
    return PagedInputs(a.q, k_cache, v_cache, table, seqlens.astype(np.int32), B, H_q, H_kv, N_q, d,
                       a.causal, a.scale, dtype)


# The five workloads the method is measured on (batch, heads, lengths, head dim,
# mask, K-row stress), with their names. Seed 0 throughout.
WORKLOADS = {
    "tiny_n256_d64": dict(B=1, H_q=1, H_kv=1, N_q=256, N_k=256, d=64, causal=False),
    "one_head_n8192_d128": dict(B=1, H_q=1, H_kv=1, N_q=8192, N_k=8192, d=128, causal=False),
    "h32_n4096_d128": dict(B=1, H_q=32, H_kv=32, N_q=4096, N_k=4096, d=128, causal=False),
    "h32_n4096_d128_causal": dict(B=1, H_q=32, H_kv=32, N_q=4096, N_k=4096, d=128, causal=True),
    "h32_n16384_d128_causal_krows": dict(B=1, H_q=32, H_kv=32, N_q=16384, N_k=16384, d=128,
                                         causal=True, k_row_frac=0.01),
    "h32_n32768_d128_causal_krows": dict(B=1, H_q=32, H_kv=32, N_q=32768, N_k=32768, d=128,
                                         causal=True, k_row_frac=0.01),
    "decode_b16_h32_kv8_n8192_d128": dict(B=16, H_q=32, H_kv=8, N_q=1, N_k=8192, d=128,
                                          causal=False),
    # head dimension 256 (the forward's widest tile plan)
    "h32_n4096_d256": dict(B=1, H_q=32, H_kv=32, N_q=4096, N_k=4096, d=256, causal=False),
    "h32_n4096_d256_causal": dict(B=1, H_q=32, H_kv=32, N_q=4096, N_k=4096, d=256, causal=True),
}


def make_workload(name: str, seed: int = 0, dtype: str = "bf16") -> AttentionInputs:
    return make_inputs(seed=seed, dtype=dtype, **WORKLOADS[name])
