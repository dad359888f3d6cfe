"""Pins of the FP8 (E4M3) pieces: the oracle's exact decode and the input
module's encoder, against a library conversion (torch.float8_e4m3fn), values
the format's definition fixes, and a brute-force nearest-value search; and
invariants of the FP8 attention reference."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_forward_gb300 import inputs as I

from oracle.fp8 import attention_reference_fp8, e4m3_to_f64

ALL = np.arange(256, dtype=np.uint8)


def test_decode_matches_library_conversion():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    lib = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).double().numpy()
    ours = oracle.e4m3_to_f64(ALL)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    fin = ~np.isnan(lib)
    assert np.array_equal(ours[fin], lib[fin]) and np.array_equal(np.signbit(ours[fin]), np.signbit(lib[fin]))


def test_decode_fixed_values():
    v = oracle.e4m3_to_f64(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x3C, 0x7E, 0x7F, 0x80, 0xB8, 0xFE, 0xFF],
                                    dtype=np.uint8))
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.5, 448.0, np.nan, -0.0, -1.0, -448.0, np.nan]
    for got, w in zip(v, want):
        assert (np.isnan(got) and np.isnan(w)) or got == w
    assert np.signbit(v[8])
    # 126 finite positive values, strictly increasing with the code
    pos = oracle.e4m3_to_f64(np.arange(0x00, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)


def _nearest_even(x, table):
    """Brute force: the finite code nearest to x, ties to the even code;
    magnitudes past 448 saturate."""
    codes = np.arange(0x7F)                     # non-negative finite codes
    vals = table[codes]
    out = np.empty(x.shape, dtype=np.uint8)
    for i, xv in enumerate(x):
        a = min(abs(xv), 448.0)
        dist = np.abs(vals - a)
        best = np.flatnonzero(dist == dist.min())
        c = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out[i] = c | (0x80 if np.signbit(xv) else 0)
    return out


def test_encoder_is_nearest_ties_to_even():
    table = oracle.e4m3_to_f64(ALL)
    rng = np.random.default_rng(40)
    pos = table[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2              # every tie between neighbours
    x = np.concatenate([rng.normal(scale=20.0, size=2000), rng.uniform(-2.0 ** -5, 2.0 ** -5, 500),
                        mids, -mids, [0.0, -0.0, 447.9, 448.0, 460.0, 464.0, 470.0, 1e30, -1e30]])
    assert np.array_equal(I.f64_to_e4m3(x), _nearest_even(x, table))


def test_encoder_matches_library_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(41)
    x = np.concatenate([rng.normal(scale=30.0, size=5000), rng.uniform(-0.02, 0.02, 2000)])
    x = x[np.abs(x) <= 448.0]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(I.f64_to_e4m3(x), lib)


def test_encoder_saturates_and_maps_nan():
    c = I.f64_to_e4m3(np.array([1e6, -1e6, 449.0, np.nan]))
    assert list(c) == [0x7E, 0xFE, 0x7E, 0x7F]


def test_e4m3_inputs_follow_their_draws():
    # the codes times the per-tensor factor stand for the FP64 deviates the bf16
    # path rounds: within half a unit in the last place (2^-4 relative) in the
    # normal range, 2^-10 * s below it
    a = I.make_inputs(1, 2, 1, 64, 96, 32, seed=5, dtype="e4m3", k_row_frac=0.02)
    b = I.make_inputs(1, 2, 1, 64, 96, 32, seed=5, dtype="bf16", k_row_frac=0.02)
    for codes, bits, s in zip((a.q, a.k, a.v), (b.q, b.k, b.v), a.descale):
        assert s > 0 and float(np.log2(s)).is_integer()
        x = oracle.e4m3_to_f64(codes) * s
        ref = oracle.bf16_to_f64(bits)            # the same deviates, rounded to BF16
        tol = np.maximum(2.0 ** -4 * np.abs(ref), 2.0 ** -10 * s) + 2.0 ** -8 * np.abs(ref)
        assert np.all(np.abs(x - ref) <= tol)
        assert np.abs(x).max() <= 448.0 * s


def test_fp8_reference_invariants():
    a = I.make_inputs(1, 2, 2, 40, 50, 16, causal=True, seed=6, dtype="e4m3")
    sq, sk, sv = a.descale
    o, lse = oracle.attention_reference_fp8(a.q, a.k, a.v, a.descale, causal=True, scale=a.scale)
    # V's factor scales O exactly and leaves LSE alone
    o2, lse2 = oracle.attention_reference_fp8(a.q, a.k, a.v, (sq, sk, 2 * sv), causal=True, scale=a.scale)
    assert np.array_equal(o2, 2 * o) and np.array_equal(lse2, lse)
    # only the product of Q's factor and the softmax scale matters
    o3, lse3 = oracle.attention_reference_fp8(a.q, a.k, a.v, (2 * sq, sk, sv), causal=True, scale=a.scale / 2)
    assert np.allclose(o3, o, rtol=0, atol=1e-14) and np.allclose(lse3, lse, rtol=0, atol=1e-12)
    # and it is the definition on the decoded values
    x = [oracle.e4m3_to_f64(c) * s for c, s in zip((a.q, a.k, a.v), a.descale)]
    o4, lse4 = oracle.attention_reference(*x, causal=True, scale=a.scale)
    assert np.array_equal(o4, o) and np.array_equal(lse4, lse)


# ---- the FP8 path's P-rounding term (oracle.p_rounding_weight / p_rounding_bound_fp8)

def test_p_rounding_weight_covers_every_reference_max():
    # E4M3 rounding of lam * p, for lam anywhere in [1, 2^8] (the kernel's lag),
    # changes it by at most lam * w(p); and the bound is reached
    from oracle.fp8 import p_rounding_weight
    p = np.concatenate([np.geomspace(2.0 ** -20, 1.0, 4001), [2.0 ** -6, 2.0 ** -10, 1.0]])
    worst = 0.0
    for lam in np.concatenate([2.0 ** np.arange(0, 9), np.geomspace(1.0, 256.0, 37)]):
        x = lam * p
        err = np.abs(e4m3_to_f64(I.f64_to_e4m3(x)) - x) / lam
        w = p_rounding_weight(p)
        assert np.all(err <= w * (1 + 1e-12)), lam
        worst = max(worst, float((err / w).max()))
    assert worst > 0.95


def _simulate_fp8(a, p_mant_bits):
    """O with the exact scores, P (against the true row max) rounded to E4M3, or
    to fewer mantissa bits when p_mant_bits < 3 (a planted mistake)."""
    from oracle.fp8 import e4m3_to_f64 as dec
    sq, sk, sv = a.descale
    q, k, v = dec(a.q)[0, 0] * sq, dec(a.k)[0, 0] * sk, dec(a.v)[0, 0] * sv
    s = a.scale * q @ k.T
    p = np.exp(s - s.max(axis=1, keepdims=True))
    l = p.sum(axis=1, keepdims=True)
    pr = dec(I.f64_to_e4m3(p))
    if p_mant_bits < 3:
        m, e = np.frexp(pr)
        step = 2.0 ** (p_mant_bits + 1)
        pr = np.ldexp(np.round(m * step) / step, e)
    return (pr @ v) / l


# (rows that sit on one or two scaled keys reach the bound; spread rows average
# their rounding errors out, so the planted mistake shows only on the former)
@pytest.mark.parametrize("n,frac,scale,seed,concentrated", [(256, 0.0, None, 3, False),
                                                          (1024, 0.02, 0.3, 5, True)])
def test_p_rounding_bound_holds_and_is_tight(n, frac, scale, seed, concentrated):
    from oracle.fp8 import p_rounding_bound_fp8
    a = I.make_inputs(1, 1, 1, n, n, 128, causal=False, seed=seed, k_row_frac=frac, scale=scale,
                      dtype="e4m3")
    o_ref, _ = attention_reference_fp8(a.q, a.k, a.v, a.descale, scale=a.scale)
    bound = p_rounding_bound_fp8(a.q, a.k, a.v, a.descale, scale=a.scale)[0, 0]
    ratio = np.abs(_simulate_fp8(a, 3) - o_ref[0, 0]) / bound
    assert ratio.max() <= 1.0
    assert ratio.max() >= (0.9 if concentrated else 0.15)
    if concentrated:
        # a planted mistake: P kept with one mantissa bit fewer than E4M3 has
        planted = np.abs(_simulate_fp8(a, 2) - o_ref[0, 0]) / bound
        assert planted.max() > 1.0


def test_p_rounding_bound_masks_like_the_definition():
    # causal: row i's bound uses keys 0..i only; a row that sees no key has 0
    from oracle.fp8 import p_rounding_bound_fp8
    a = I.make_inputs(1, 2, 1, 40, 24, 128, causal=True, seed=2, dtype="e4m3")
    full = p_rounding_bound_fp8(a.q, a.k, a.v, a.descale, causal=True, scale=a.scale)
    assert np.all(full[:, :, :16] == 0.0)            # N_q > N_k: rows 0..15 see no key
    # row 16 sees key 0 only: p = 1, weight 2^-4, l = 1
    v0 = np.abs(e4m3_to_f64(a.v[0, 0, 0]) * a.descale[2])
    assert np.allclose(full[0, 0, 16], 2.0 ** -4 * v0, rtol=1e-12)
