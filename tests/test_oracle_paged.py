"""Pins of the paged-cache decode oracle against caches this test builds itself:
contiguous keys scattered into pages of 128 by a permutation the test draws,
then the paged result must equal the definition on the contiguous prefix
exactly (the same FP64 arithmetic on the same values)."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_forward_gb300 import inputs as I


def _scatter(k, v, lens, rng, spare=2):
    """Pages [P][H_kv][128][d] holding sequence b's keys in order, pages shuffled,
    garbage in the tails, spare pages and unused table entries."""
    B, H_kv, n, d = k.shape
    used = [(L + 127) // 128 for L in lens]
    P = sum(used) + spare
    perm = rng.permutation(P)
    kc = rng.normal(size=(P, H_kv, 128, d))
    vc = rng.normal(size=(P, H_kv, 128, d))
    max_pages = max(max(used), 1)
    table = rng.integers(0, P, size=(B, max_pages)).astype(np.int32)
    s = 0
    for b in range(B):
        for j in range(used[b]):
            pg = perm[s]
            s += 1
            table[b, j] = pg
            lo, hi = j * 128, min((j + 1) * 128, lens[b])
            kc[pg, :, :hi - lo] = k[b, :, lo:hi]
            vc[pg, :, :hi - lo] = v[b, :, lo:hi]
    return kc, vc, table


@pytest.mark.parametrize("causal", [False, True])
def test_paged_equals_contiguous_prefix(causal):
    rng = np.random.default_rng(5)
    B, H_q, H_kv, n_q, d = 4, 4, 2, 3, 8
    lens = [1, 128, 129, 300]
    k = rng.normal(size=(B, H_kv, 300, d))
    v = rng.normal(size=(B, H_kv, 300, d))
    q = rng.normal(size=(B, H_q, n_q, d))
    kc, vc, table = _scatter(k, v, lens, rng)
    o, lse = oracle.paged_attention_reference(q, kc, vc, table, np.array(lens), causal=causal, scale=0.3)
    for b, L in enumerate(lens):
        ob, lb = oracle.attention_reference(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], causal=causal,
                                            scale=0.3)
        assert np.array_equal(o[b], ob[0]) and np.array_equal(lse[b], lb[0])


def test_paged_ignores_tails_and_unused_entries():
    rng = np.random.default_rng(6)
    q = rng.normal(size=(2, 2, 1, 4))
    k = rng.normal(size=(2, 1, 200, 4))
    v = rng.normal(size=(2, 1, 200, 4))
    kc, vc, table = _scatter(k, v, [70, 200], rng)
    o1, l1 = oracle.paged_attention_reference(q, kc, vc, table, np.array([70, 200]))
    # overwrite everything no key of a sequence lives in
    kc2, vc2, table2 = kc.copy(), vc.copy(), table.copy()
    kc2[table[0, 0], :, 70:] = 1e6
    vc2[table[1, 1], :, 72:] = -1e6
    owned = {int(table[0, 0]), int(table[1, 0]), int(table[1, 1])}
    for pg in range(kc.shape[0]):
        if pg not in owned:
            kc2[pg] = 7.0
            vc2[pg] = 7.0
    table2[0, 1] = (int(table[0, 1]) + 1) % kc.shape[0]
    o2, l2 = oracle.paged_attention_reference(q, kc2, vc2, table2, np.array([70, 200]))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_empty_sequence():
    rng = np.random.default_rng(7)
    q = rng.normal(size=(2, 2, 2, 4))
    k = rng.normal(size=(2, 2, 130, 4))
    kc, vc, table = _scatter(k, k, [0, 130], rng)
    o, lse = oracle.paged_attention_reference(q, kc, vc, table, np.array([0, 130]))
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_make_paged_layout():
    # the generator's pages hold make_inputs' own draws of K and V, in order
    p = I.make_paged(3, 4, 2, 2, [0, 129, 300], 64, seed=1)
    a = I.make_inputs(3, 4, 2, 2, 3 * 128, 64, seed=1)
    assert np.array_equal(p.q, a.q)
    for b, L in enumerate([0, 129, 300]):
        assert np.array_equal(oracle.gather_sequence(p.k_cache, p.block_table, b, L), a.k[b, :, :L])
        assert np.array_equal(oracle.gather_sequence(p.v_cache, p.block_table, b, L), a.v[b, :, :L])
    # every page a sequence uses is its own
    owned = [int(p.block_table[b, j]) for b, L in enumerate([0, 129, 300]) for j in range((L + 127) // 128)]
    assert len(owned) == len(set(owned)) == 5
