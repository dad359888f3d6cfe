"""Pins of the FP64 backward oracle against things other than itself: central
finite differences of the forward oracle (the gradient of sum(dO * O)), closed
forms and invariants of the softmax Jacobian."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_forward_gb300 import inputs as I

SHAPES = [
    # (B, H_q, H_kv, N_q, N_k, d, causal)
    (1, 2, 1, 5, 7, 4, True),      # GQA, N_q < N_k
    (1, 2, 2, 6, 4, 3, False),
    (2, 4, 2, 3, 5, 4, True),
    (1, 1, 1, 6, 3, 4, True),      # N_q > N_k: the first rows see no key
]


def _random(shape, seed):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(B, Hq, Nq, d)), rng.normal(size=(B, Hkv, Nk, d)),
            rng.normal(size=(B, Hkv, Nk, d)), rng.normal(size=(B, Hq, Nq, d)), causal)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gradients_match_central_differences(shape):
    q, k, v, do, causal = _random(shape, 11)
    scale = 0.7
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=causal, scale=scale)
    h = 1e-5
    for x, g in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            keep = x[idx]
            x[idx] = keep + h
            up = oracle.forward_loss(q, k, v, do, causal=causal, scale=scale)
            x[idx] = keep - h
            dn = oracle.forward_loss(q, k, v, do, causal=causal, scale=scale)
            x[idx] = keep
            fd[idx] = (up - dn) / (2 * h)
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-8)


def test_equal_value_rows_give_no_query_or_key_gradient():
    # O = c for every row whatever P is, so S (hence Q, K) cannot move the loss
    q, k, v, do, _ = _random((1, 2, 1, 6, 9, 4, False), 12)
    v[:] = v[:, :, :1]
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=False, scale=0.5)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.abs(dv).max() > 0.1


def test_zero_upstream_gradient():
    q, k, v, do, _ = _random((1, 1, 1, 4, 4, 4, True), 13)
    grads = oracle.attention_backward(q, k, v, np.zeros_like(do), causal=True)
    assert all(np.abs(x).max() == 0.0 for x in grads)


def test_query_gradient_ignores_a_shift_of_all_keys():
    # rows of dS sum to zero (softmax Jacobian), so dQ = scale dS K is blind to K + u
    q, k, v, do, _ = _random((1, 2, 2, 5, 8, 4, False), 14)
    dq, dk, _ = oracle.attention_backward(q, k, v, do, causal=False, scale=0.3)
    u = np.array([0.5, -1.0, 2.0, 0.25])
    q2, k2 = q.copy(), k + u
    # shifting K also shifts the scores by q . u per row: a per-row constant, so P is unchanged
    dq2, dk2, _ = oracle.attention_backward(q2, k2, v, do, causal=False, scale=0.3)
    np.testing.assert_allclose(dq2, dq, atol=1e-12)


def test_gqa_equals_repeated_heads_summed():
    q, k, v, do, _ = _random((1, 4, 2, 5, 6, 4, True), 15)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=True, scale=0.6)
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    dq_m, dk_m, dv_m = oracle.attention_backward(q, kr, vr, do, causal=True, scale=0.6)
    np.testing.assert_allclose(dq, dq_m, atol=1e-13)
    np.testing.assert_allclose(dk, dk_m.reshape(1, 2, 2, 6, 4).sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(dv, dv_m.reshape(1, 2, 2, 6, 4).sum(axis=2), atol=1e-13)


def test_bits_inputs_widen_exactly():
    # BF16 bit patterns and their float64 values give the same gradients
    a = I.make_inputs(1, 2, 1, 7, 9, 8, causal=True, seed=3)
    do = I.grad_output(a, seed=3)
    g_bits = oracle.attention_backward(a.q, a.k, a.v, do, causal=True, scale=a.scale)
    w = oracle.to_f64
    g_f64 = oracle.attention_backward(w(a.q), w(a.k), w(a.v), w(do), causal=True, scale=a.scale)
    for x, y in zip(g_bits, g_f64):
        assert np.array_equal(x, y)


# ---- the backward tolerance (backward_error_terms), pinned by simulating on
# the CPU each rounding a 16-bit backward does, one at a time: P rounded before
# dV = P^T dO, dS rounded before dQ = scale dS K and dK = scale dS^T Q, and O
# rounded before D = rowsum(dO * O). Each effect must lie within u times its own
# term (sound), and reach at least 5 % of it somewhere (not vacuously loose).

def _round_bf16(x):
    return I.bf16_bits_to_f32(I.f64_to_bf16_bits(x)).astype(np.float64)


def _simulated_gradients(a, do, rounded):
    """dQ, dK, dV in FP64 with one intermediate ("P", "dS" or "O") rounded to BF16."""
    from oracle.backward import _probabilities
    q, k, v, g = (oracle.to_f64(x) for x in (a.q, a.k, a.v, do))
    G = a.H_q // a.H_kv
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(a.B):
        for h in range(a.H_q):
            hk = h // G
            p = _probabilities(q[b, h], k[b, hk], a.N_q, a.N_k, a.causal, a.scale)
            o = p @ v[b, hk]
            dv[b, hk] += (_round_bf16(p) if rounded == "P" else p).T @ g[b, h]
            dd = (g[b, h] * (_round_bf16(o) if rounded == "O" else o)).sum(axis=1, keepdims=True)
            ds = p * (g[b, h] @ v[b, hk].T - dd)
            if rounded == "dS":
                ds = _round_bf16(ds)
            dq[b, h] = a.scale * ds @ k[b, hk]
            dk[b, hk] += a.scale * ds.T @ q[b, h]
    return dq, dk, dv


BOUND_SHAPES = [(1, 2, 1, 24, 40, 8, True), (1, 1, 1, 32, 32, 16, False), (2, 2, 2, 20, 12, 8, True)]


@pytest.mark.parametrize("shape", BOUND_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_error_terms_cover_each_rounding(shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=3)
    do = I.grad_output(a, seed=3)
    u = 2.0 ** -8
    ref = oracle.attention_backward(a.q, a.k, a.v, do, causal=causal, scale=a.scale)
    t = oracle.backward_error_terms(a.q, a.k, a.v, do, causal=causal, scale=a.scale, parts=True)
    checks = {"P": [(2, "dv_p")], "dS": [(0, "dq_ds"), (1, "dk_ds")], "O": [(0, "dq_d"), (1, "dk_d")]}
    for rounded, pairs in checks.items():
        sim = _simulated_gradients(a, do, rounded)
        for i, part in pairs:
            err = np.abs(sim[i] - ref[i])
            bound = u * t[part]
            ratio = err / np.where(bound > 0, bound, 1.0)
            assert np.all(err[bound == 0] < 1e-15), (rounded, part)
            assert ratio.max() <= 1.0, (rounded, part, ratio.max())
            assert ratio.max() >= 0.05, (rounded, part, ratio.max())
        # the gradients this rounding does not touch stay exact
        for i in set(range(3)) - {i for i, _ in pairs}:
            assert np.allclose(sim[i], ref[i], rtol=0, atol=1e-12)


def test_error_terms_sum_of_parts():
    a = I.make_inputs(1, 2, 1, 9, 13, 4, causal=True, seed=4)
    do = I.grad_output(a, seed=4)
    tq, tk, tv = oracle.backward_error_terms(a.q, a.k, a.v, do, causal=True, scale=a.scale)
    t = oracle.backward_error_terms(a.q, a.k, a.v, do, causal=True, scale=a.scale, parts=True)
    assert np.array_equal(tq, t["dq_ds"] + t["dq_d"]) and np.array_equal(tk, t["dk_ds"] + t["dk_d"])
    assert np.array_equal(tv, t["dv_p"])


# ---- closed forms of the definition's gradients

def test_single_key_closed_form():
    # one key: P = 1 for every row, so O = V_0 whatever Q and K are: dQ = dK = 0
    # and dV_0 sums dO over every row of every query head that reads it
    rng = np.random.default_rng(21)
    q, k, v = rng.normal(size=(2, 4, 5, 3)), rng.normal(size=(2, 2, 1, 3)), rng.normal(size=(2, 2, 1, 3))
    do = rng.normal(size=(2, 4, 5, 3))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale=0.9)
    assert np.allclose(dq, 0, atol=1e-14) and np.allclose(dk, 0, atol=1e-14)
    want = do.reshape(2, 2, 2, 5, 3).sum(axis=(2, 3))[:, :, None, :]
    assert np.allclose(dv, want, rtol=0, atol=1e-12)


def test_zero_queries_closed_form():
    # Q = 0: every row attends uniformly, P = 1/N_k, so dV_j = (1/N_k) sum_i dO_i
    # for every key j; dK = scale dS^T Q = 0
    rng = np.random.default_rng(22)
    n_q, n_k, d = 6, 7, 4
    q = np.zeros((1, 1, n_q, d))
    k, v, do = rng.normal(size=(1, 1, n_k, d)), rng.normal(size=(1, 1, n_k, d)), rng.normal(size=(1, 1, n_q, d))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale=0.5)
    assert np.allclose(dk, 0, atol=1e-14)
    assert np.allclose(dv[0, 0], np.tile(do[0, 0].sum(axis=0) / n_k, (n_k, 1)), rtol=0, atol=1e-12)
    # dQ_i = scale sum_j P_ij (dP_ij - D_i) k_j with P uniform and D_i = dO_i . mean(V)
    vbar = v[0, 0].mean(axis=0)
    dp = do[0, 0] @ v[0, 0].T
    want = 0.5 / n_k * ((dp - (do[0, 0] @ vbar)[:, None]) @ k[0, 0])
    assert np.allclose(dq[0, 0], want, rtol=0, atol=1e-12)


def test_rows_that_see_no_key_contribute_nothing():
    # causal with N_q > N_k: the first N_q - N_k rows see no key; their dQ is 0 and
    # removing them (with their dO) leaves dK and dV unchanged
    rng = np.random.default_rng(23)
    q, k, v = rng.normal(size=(1, 2, 7, 4)), rng.normal(size=(1, 1, 4, 4)), rng.normal(size=(1, 1, 4, 4))
    do = rng.normal(size=(1, 2, 7, 4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=True, scale=0.6)
    assert np.all(dq[:, :, :3] == 0)
    dq2, dk2, dv2 = oracle.attention_backward(q[:, :, 3:], k, v, do[:, :, 3:], causal=True, scale=0.6)
    assert np.allclose(dk, dk2, rtol=0, atol=1e-12) and np.allclose(dv, dv2, rtol=0, atol=1e-12)
    assert np.allclose(dq[:, :, 3:], dq2, rtol=0, atol=1e-12)
