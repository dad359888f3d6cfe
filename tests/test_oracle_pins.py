"""Pins of the FP64 oracle against what the pages and the mathematics fix.

Each test below would fail for a plausible slip in the oracle: a dropped
scale, a missing max subtraction, a wrong sign in the rescale factor, a wrong
GQA head map, a transposed operand, an off-by-one in the causal mask, or a
wrong log in the LSE.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from oracle.attention import bf16_to_f64
from exact_tiled_attention_forward_gb300 import inputs as I

from conftest import read_golden


def _bits(x):
    """float array -> bf16 bit patterns (values chosen exactly representable)."""
    return I.f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


# ---- the toy run (page 3, Step 3) ------------------------------------------------

def test_toy_online_softmax_every_split():
    g = {r[0]: r[1:] for r in read_golden("toy_online_softmax.txt")}
    scores = [float(x) for x in g["scores"]]
    want_w = [float(x) for x in g["weights"]]
    eye = np.eye(4)
    for cut in range(1, 4):  # "two blocks": every split point gives the same result
        m, l, o = oracle.online_softmax_blocks([scores[:cut], scores[cut:]],
                                               [eye[:cut], eye[cut:]])
        assert m == float(g["max"][0])
        assert round(l, 3) == float(g["sum"][0])
        assert l == pytest.approx(1 + math.exp(-1) + math.exp(-2) + math.exp(-3), abs=1e-15)
        w = o / l  # V = I: the output row is the weight vector
        assert [round(x, 4) for x in w] == want_w
    # one pass over all four gives the same state
    m1, l1, o1 = oracle.online_softmax_blocks([scores], [eye])
    assert (m1, l1) == (3.0, pytest.approx(l, abs=1e-15))


def test_toy_run_through_attention_reference():
    # scores 2, 1, 0, 3 as one query against four keys (scale 1, d = 4, V = I)
    q = _bits([[[[1, 0, 0, 0]]]])
    k = _bits([[[[2, 0, 0, 0], [1, 0, 0, 0], [0, 0, 0, 0], [3, 0, 0, 0]]]])
    v = _bits([[np.eye(4)]])
    o, lse = oracle.attention_reference(q, k, v, scale=1.0)
    g = {r[0]: r[1:] for r in read_golden("toy_online_softmax.txt")}
    assert [round(x, 4) for x in o[0, 0, 0]] == [float(x) for x in g["weights"]]
    assert lse[0, 0, 0] == pytest.approx(3 + math.log(1 + math.exp(-1) + math.exp(-2) + math.exp(-3)),
                                         abs=1e-14)


# ---- softmax rows, brute force ----------------------------------------------------

def test_rows_of_p_are_a_distribution():
    # V = identity (N_k = d): O equals P itself
    a = I.make_inputs(1, 2, 1, 37, 64, 64, seed=3)
    v = _bits(np.broadcast_to(np.eye(64), (1, 1, 64, 64)))
    for causal in (False, True):
        p, _ = oracle.attention_reference(a.q, a.k, v, causal=causal, scale=a.scale)
        assert (p >= 0).all()
        np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
        if causal:  # row i may only weight keys 0 .. i + N_k - N_q
            for i in range(37):
                assert np.all(p[0, :, i, i + 64 - 37 + 1:] == 0)


@pytest.mark.parametrize("shape,causal", [
    ((1, 1, 1, 5, 7, 4), False),
    ((1, 2, 2, 9, 9, 8), True),
    ((2, 4, 2, 6, 11, 3), True),    # GQA, N_q < N_k, odd d
    ((1, 2, 1, 13, 5, 8), True),    # N_q > N_k: leading rows see no key
    ((1, 1, 1, 16, 16, 8), False),
])
def test_brute_force_agrees(shape, causal):
    B, Hq, Hkv, Nq, Nk, d = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=11)
    o, lse = oracle.attention_reference(a.q, a.k, a.v, causal=causal, scale=a.scale)
    ob, lb = oracle.brute_force_attention(bf16_to_f64(a.q).tolist(), bf16_to_f64(a.k).tolist(),
                                          bf16_to_f64(a.v).tolist(), causal=causal, scale=a.scale)
    np.testing.assert_allclose(o, np.array(ob), atol=1e-12, rtol=0)
    lb = np.array(lb)
    assert np.array_equal(np.isinf(lse), np.isinf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], atol=1e-12, rtol=0)
    if Nq > Nk and causal:
        # rows 0 .. Nq-Nk-1 see no key: O = 0, LSE = -inf
        assert np.all(o[:, :, : Nq - Nk] == 0) and np.all(np.isneginf(lse[:, :, : Nq - Nk]))


# ---- tiled online softmax vs materialised (page 2 harness) ------------------------

@pytest.mark.parametrize("block", [16, 32, 64, 128])
def test_tiled_matches_materialised_page2_harness(block):
    # "Flash Attention Mechanics", "The Tiling Algorithm": seed 0, seq 1024, d 64,
    # blocks 16..128, max abs error between tiled and standard. Exact in algebra;
    # in FP64 the two orders agree to rounding (reading: <= 1e-12, not bit-exact).
    a = I.make_inputs(1, 1, 1, 1024, 1024, 64, seed=0)
    o_ref, l_ref = oracle.attention_reference(a.q, a.k, a.v, scale=a.scale)
    o_t, l_t = oracle.attention_tiled_online(a.q, a.k, a.v, block, block, scale=a.scale)
    assert np.max(np.abs(o_ref - o_t)) <= 1e-12
    assert np.max(np.abs(l_ref - l_t)) <= 1e-12


def test_tiled_matches_materialised_causal_ragged_gqa():
    a = I.make_inputs(2, 4, 2, 100, 133, 16, causal=True, seed=5, k_row_frac=0.05)
    o_ref, l_ref = oracle.attention_reference(a.q, a.k, a.v, causal=True, scale=a.scale)
    for bq, bk in [(7, 13), (32, 32), (128, 64)]:
        o_t, l_t = oracle.attention_tiled_online(a.q, a.k, a.v, bq, bk, causal=True, scale=a.scale)
        np.testing.assert_allclose(o_t, o_ref, atol=1e-12, rtol=0)
        np.testing.assert_allclose(l_t, l_ref, atol=1e-12, rtol=0)


# ---- closed forms -------------------------------------------------------------------

def test_zero_query_gives_mean_of_values():
    a = I.make_inputs(1, 1, 1, 8, 50, 32, seed=2)
    q = np.zeros_like(a.q)
    o, lse = oracle.attention_reference(q, a.k, a.v, scale=a.scale)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(bf16_to_f64(a.v[0, 0]).mean(0), (8, 32)),
                               atol=1e-14)
    np.testing.assert_allclose(lse, math.log(50), atol=1e-14)


def test_single_key():
    a = I.make_inputs(1, 1, 1, 6, 1, 16, seed=4)
    o, lse = oracle.attention_reference(a.q, a.k, a.v, scale=0.3)
    np.testing.assert_array_equal(o[0, 0], np.broadcast_to(bf16_to_f64(a.v[0, 0, 0]), (6, 16)))
    s00 = 0.3 * bf16_to_f64(a.q[0, 0]) @ bf16_to_f64(a.k[0, 0, 0])
    np.testing.assert_allclose(lse[0, 0], s00, atol=1e-14)


def test_equal_keys_give_mean_and_shifted_lse():
    a = I.make_inputs(1, 1, 1, 5, 40, 8, seed=6)
    k = np.broadcast_to(a.k[:, :, :1], a.k.shape).copy()
    o, lse = oracle.attention_reference(a.q, k, a.v, scale=a.scale)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(bf16_to_f64(a.v[0, 0]).mean(0), (5, 8)),
                               atol=1e-14)
    s = a.scale * bf16_to_f64(a.q[0, 0]) @ bf16_to_f64(a.k[0, 0, 0])
    np.testing.assert_allclose(lse[0, 0], s + math.log(40), atol=1e-13)


def test_constant_values_and_dominant_key():
    a = I.make_inputs(1, 1, 1, 4, 30, 8, seed=7)
    v = _bits(np.full((1, 1, 30, 8), 1.5))
    o, _ = oracle.attention_reference(a.q, a.k, v, scale=a.scale)
    np.testing.assert_allclose(o, 1.5, atol=1e-14)
    # one key far larger than the rest: O is that key's value row
    q = _bits(np.tile([[1.0] + [0.0] * 7], (4, 1))[None, None])
    k = np.zeros((1, 1, 30, 8))
    k[0, 0, 17, 0] = 64.0     # score 64 vs 0 (scale 1): other weights ~ e^-64
    o, lse = oracle.attention_reference(q, _bits(k), a.v, scale=1.0)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(bf16_to_f64(a.v[0, 0, 17]), (4, 8)),
                               atol=30 * math.exp(-64) * 8)
    np.testing.assert_allclose(lse, 64.0, atol=1e-14)


# ---- invariants ----------------------------------------------------------------------

def test_key_shift_moves_lse_only():
    # K entries and the shift u are multiples of 1/4 below 8 in magnitude, so K + u
    # is exact in bfloat16 and both problems go through the oracle unchanged.
    rng = np.random.default_rng(1)
    a = I.make_inputs(1, 1, 1, 9, 21, 8, seed=8)
    k = rng.integers(-12, 13, size=(1, 1, 21, 8)) / 4.0
    u = np.array([0.5, -1.0, 0.25, 2.0, 0.0, -0.5, 1.0, 0.75])
    o0, l0 = oracle.attention_reference(a.q, _bits(k), a.v, scale=a.scale)
    o1, l1 = oracle.attention_reference(a.q, _bits(k + u), a.v, scale=a.scale)
    np.testing.assert_allclose(o1, o0, atol=1e-13)
    np.testing.assert_allclose(l1[0, 0], l0[0, 0] + a.scale * bf16_to_f64(a.q[0, 0]) @ u, atol=1e-12)


def test_joint_key_value_permutation():
    a = I.make_inputs(1, 2, 2, 10, 33, 8, seed=9)
    perm = np.random.default_rng(0).permutation(33)
    o0, l0 = oracle.attention_reference(a.q, a.k, a.v, scale=a.scale)
    o1, l1 = oracle.attention_reference(a.q, a.k[:, :, perm], a.v[:, :, perm], scale=a.scale)
    np.testing.assert_allclose(o1, o0, atol=1e-14)
    np.testing.assert_allclose(l1, l0, atol=1e-13)


def test_causal_row_equals_noncausal_prefix():
    a = I.make_inputs(1, 1, 1, 24, 24, 8, seed=10)
    oc, lc = oracle.attention_reference(a.q, a.k, a.v, causal=True, scale=a.scale)
    np.testing.assert_array_equal(oc[0, 0, 0], bf16_to_f64(a.v[0, 0, 0]))  # row 0 = V_0
    for i in (0, 1, 7, 23):
        o, l = oracle.attention_reference(a.q[:, :, i:i + 1], a.k[:, :, : i + 1], a.v[:, :, : i + 1],
                                          scale=a.scale)
        np.testing.assert_allclose(oc[0, 0, i], o[0, 0, 0], atol=1e-14)
        np.testing.assert_allclose(lc[0, 0, i], l[0, 0, 0], atol=1e-14)


def test_gqa_equals_mha_with_repeated_kv():
    a = I.make_inputs(2, 6, 2, 7, 19, 8, causal=True, seed=12)
    o, l = oracle.attention_reference(a.q, a.k, a.v, causal=True, scale=a.scale)
    k_rep = np.repeat(a.k, 3, axis=1)
    v_rep = np.repeat(a.v, 3, axis=1)
    o2, l2 = oracle.attention_reference(a.q, k_rep, v_rep, causal=True, scale=a.scale)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(l, l2)


def test_heads_and_batches_independent():
    a = I.make_inputs(2, 3, 3, 8, 12, 8, seed=13)
    o, l = oracle.attention_reference(a.q, a.k, a.v, scale=a.scale)
    for b, h in itertools.product(range(2), range(3)):
        o1, l1 = oracle.attention_reference(a.q[b:b + 1, h:h + 1], a.k[b:b + 1, h:h + 1],
                                            a.v[b:b + 1, h:h + 1], scale=a.scale)
        np.testing.assert_array_equal(o[b, h], o1[0, 0])
        np.testing.assert_array_equal(l[b, h], l1[0, 0])


def test_rows_subset_matches_full():
    a = I.make_inputs(1, 4, 2, 300, 280, 16, causal=True, seed=14)
    o, l = oracle.attention_reference(a.q, a.k, a.v, causal=True, scale=a.scale)
    rows = np.array([0, 1, 19, 20, 21, 150, 299])
    for h in (0, 3):
        o1, l1 = oracle.attention_rows(a.q, a.k, a.v, 0, h, rows, causal=True, scale=a.scale)
        np.testing.assert_allclose(o1, o[0, h, rows], atol=1e-14)
        assert np.array_equal(np.isneginf(l1), np.isneginf(l[0, h, rows]))
        fin = np.isfinite(l1)
        np.testing.assert_allclose(l1[fin], l[0, h, rows][fin], atol=1e-14)


# ---- split-KV merge ------------------------------------------------------------------

@pytest.mark.parametrize("cuts", [[64], [1, 2, 100], [0, 50, 50, 127], [30, 60, 90]])
def test_merge_of_key_ranges_equals_unsplit(cuts):
    a = I.make_inputs(1, 1, 1, 12, 128, 16, causal=True, seed=15, k_row_frac=0.05)
    o_ref, l_ref = oracle.attention_reference(a.q, a.k, a.v, causal=True, scale=a.scale)
    qf = bf16_to_f64(a.q[0, 0])
    kf = bf16_to_f64(a.k[0, 0])
    vf = bf16_to_f64(a.v[0, 0])
    bounds = [0] + cuts + [128]
    ms, ls, os_ = [], [], []
    vis = oracle.visible_key_count(np.arange(12), 12, 128, True)
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        s = a.scale * qf @ kf[lo:hi].T
        s = np.where(np.arange(lo, hi)[None, :] < vis[:, None], s, -np.inf)
        m = s.max(1) if hi > lo else np.full(12, -np.inf)
        ref = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(s - ref[:, None])
        ms.append(m)
        ls.append(e.sum(1))
        os_.append(e @ vf[lo:hi])
    o, l = oracle.merge_partials(ms, ls, os_)
    np.testing.assert_allclose(o, o_ref[0, 0], atol=1e-13)
    np.testing.assert_allclose(l, l_ref[0, 0], atol=1e-13)
