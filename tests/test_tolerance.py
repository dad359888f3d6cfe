"""Pins of the element-wise O tolerance the GPU parity tests use
(helpers.elementwise_bound), checked on the CPU without any kernel.

The bound claims: when each probability is rounded to the 16-bit type before
the P V product and the output is rounded to the same type, every element of O
stays within half_spacing(|O_ref| + u A) + u A of the exact result. Here the
two roundings are simulated in FP64 on inputs whose rows sit on a few scaled
keys (large |O|), and the bound must hold (without its 1e-2 floor), come close
to being reached (it is not loose), and fail when a rounding is made coarser
than the type the bound names (a planted mistake).
"""
import numpy as np
import pytest

import oracle
from oracle.attention import bf16_to_f64
from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import abs_values, elementwise_bound, half_spacing


def _round_bits(x, mant_bits):
    """Round FP64 values to nearest (ties to even) with `mant_bits` stored
    mantissa bits, exponent range unlimited (no subnormals needed here)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                              # x = m 2^e, 0.5 <= |m| < 1
    scale = 2.0 ** (mant_bits + 1)
    return np.ldexp(np.round(m * scale) / scale, e)   # np.round: half to even


def test_half_spacing_matches_the_types():
    torch = pytest.importorskip("torch")
    xs = np.array([1e-3, 0.3, 0.75, 1.0, 1.5, 2.4, 3.99, 4.0, 100.0, 60000.0])
    for x in xs:
        # spacing above x, from the types themselves
        b = torch.tensor([x], dtype=torch.float64).to(torch.bfloat16)
        b_next = torch.nextafter(b.float(), torch.tensor([np.inf])).to(torch.bfloat16)
        lo = float(b.float()) if float(b.float()) <= x else None
        if lo is not None and float(b_next.float()) > lo:
            step = float(b_next.float()) - lo
            if np.frexp(lo)[1] == np.frexp(x)[1]:
                assert half_spacing(x, "bf16") == step / 2, x
        h = np.float16(x)
        if float(h) <= x and np.isfinite(h):
            step = float(np.nextafter(h, np.float16(np.inf))) - float(h)
            if np.frexp(float(h))[1] == np.frexp(x)[1]:
                assert half_spacing(x, "f16") == step / 2, x
    assert half_spacing(1.0) == 2.0 ** -8 and half_spacing(2.4) == 2.0 ** -7
    assert half_spacing(1.0, "f16") == 2.0 ** -11
    assert half_spacing(1e-9, "f16") == 2.0 ** -25    # FP16 subnormal spacing 2^-24


def _simulate(a, p_bits, o_bits):
    """O with P rounded to p_bits and O rounded to o_bits stored mantissa bits."""
    q, k, v = bf16_to_f64(a.q)[0, 0], bf16_to_f64(a.k)[0, 0], bf16_to_f64(a.v)[0, 0]
    s = a.scale * q @ k.T
    p = np.exp(s - s.max(axis=1, keepdims=True))
    l = p.sum(axis=1, keepdims=True)
    o = (_round_bits(p, p_bits) @ v) / l
    return _round_bits(o, o_bits)


@pytest.fixture(scope="module")
def concentrated():
    # 2 % of the keys scaled by 8 and a larger scale: many rows put most of their
    # weight on one or two keys, so |O| reaches 2-3 and A ~ |O|
    a = I.make_inputs(1, 1, 1, 256, 512, 64, causal=False, seed=7, k_row_frac=0.02, scale=0.3)
    o_ref, _ = oracle.attention_reference(a.q, a.k, a.v, causal=False, scale=a.scale)
    a_ref, _ = oracle.attention_reference(a.q, a.k, abs_values(a.v), causal=False, scale=a.scale)
    return a, o_ref[0, 0], a_ref[0, 0]


def test_bound_holds_and_is_nearly_reached(concentrated):
    a, o_ref, a_ref = concentrated
    assert np.abs(o_ref).max() > 2.0                     # the regime where 1e-2 is not enough
    got = _simulate(a, 7, 7)                             # BF16: 7 stored mantissa bits
    ratio = np.abs(got - o_ref) / elementwise_bound(o_ref, a_ref, "bf16", floor=0.0)
    assert ratio.max() <= 1.0
    assert ratio.max() >= 0.5                             # the bound is not loose


def test_bound_catches_coarser_roundings(concentrated):
    a, o_ref, a_ref = concentrated
    bound = elementwise_bound(o_ref, a_ref, "bf16", floor=0.0)
    for p_bits, o_bits in ((6, 7), (7, 6)):              # one bit short in P, or in O
        got = _simulate(a, p_bits, o_bits)
        assert (np.abs(got - o_ref) / bound).max() > 1.0, (p_bits, o_bits)


def test_fp16_bound_holds(concentrated):
    a, o_ref, a_ref = concentrated
    got = _simulate(a, 10, 10)                           # FP16: 10 stored mantissa bits
    ratio = np.abs(got - o_ref) / elementwise_bound(o_ref, a_ref, "f16", floor=0.0)
    assert 0.3 <= ratio.max() <= 1.0
