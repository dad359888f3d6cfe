"""GPU parity of fa_decode_paged (decode over a paged K/V cache, through the C
ABI) against the FP64 oracle (each sequence's keys read out of its pages, then
the definition), element by element; and bit-identity with fa_forward over the
same keys stored contiguously (the same kernel and plan)."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import compare, to_dev, abs_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import exact_tiled_attention_forward_gb300 as fa
    from exact_tiled_attention_forward_gb300 import build
    build.build()
    fa.lib()
    return fa


GUARD = 4096


def _run(fa, p):
    """fa_decode_paged with O and LSE inside canary margins that must stay untouched."""
    import torch
    q, kc, vc = to_dev(p.q), to_dev(p.k_cache), to_dev(p.v_cache)
    table = torch.from_numpy(p.block_table).cuda()
    lens = torch.from_numpy(p.seqlens).cuda()
    n = p.q.size
    ob = torch.full((n + 2 * GUARD,), -7.0, dtype=q.dtype, device="cuda")
    lb = torch.full((n // p.d + 2 * GUARD,), -7.0, dtype=torch.float32, device="cuda")
    o = ob[GUARD:GUARD + n].view(q.shape)
    lse = lb[GUARD:GUARD + n // p.d].view(p.B, p.H_q, p.N_q)
    fa.fa_decode_paged(q, kc, vc, table, lens, causal=p.causal, scale=p.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    for buf in (ob, lb):
        assert bool(torch.all(buf[:GUARD] == -7.0)) and bool(torch.all(buf[-GUARD:] == -7.0))
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _oracle(p):
    """(O, LSE, A): the oracle's O and LSE, and A = the same attention of |V|."""
    o, lse = oracle.paged_attention_reference(p.q, p.k_cache, p.v_cache, p.block_table, p.seqlens,
                                              causal=p.causal, scale=p.scale)
    o_abs, _ = oracle.paged_attention_reference(p.q, p.k_cache, abs_values(p.v_cache), p.block_table,
                                                p.seqlens, causal=p.causal, scale=p.scale)
    return o, lse, o_abs


CASES = [
    # (B, H_q, H_kv, N_q, seqlens, d, causal)
    (3, 4, 2, 1, [0, 1, 300], 128, False),            # an empty sequence, one key, a ragged page
    (4, 8, 2, 4, [127, 128, 129, 1000], 128, True),   # GQA 4 x 4 rows = 16, page boundaries
    (2, 16, 1, 1, [5000, 64], 64, False),             # MQA, d = 64, very unequal lengths
    (5, 4, 4, 3, [0, 3, 2, 700, 1], 128, True),       # causal rows that see no key (N_q > length)
    (16, 32, 8, 1, [8192] * 15 + [100], 128, False),  # the decode batch, one short sequence
    (8, 8, 8, 2, [4100, 4096, 1, 0, 3000, 129, 256, 8000], 128, True),
]


@pytest.mark.parametrize("cluster_merge", [True, False], ids=["cluster", "kernel"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"b{c[0]}h{c[1]}kv{c[2]}q{c[3]}d{c[5]}" + ("c" if c[6] else ""))
def test_paged_parity(fa, case, cluster_merge, monkeypatch):
    monkeypatch.setenv("FA_CLUSTER_MERGE", "1" if cluster_merge else "0")
    B, Hq, Hkv, Nq, lens, d, causal = case
    p = I.make_paged(B, Hq, Hkv, Nq, lens, d, causal=causal, seed=31)
    o, lse = _run(fa, p)
    compare(o, lse, *_oracle(p))


@pytest.mark.parametrize("case", [CASES[1], CASES[3]], ids=["gqa", "short"])
def test_paged_parity_fp16(fa, case):
    B, Hq, Hkv, Nq, lens, d, causal = case
    p = I.make_paged(B, Hq, Hkv, Nq, lens, d, causal=causal, seed=32, dtype="f16")
    o, lse = _run(fa, p)
    compare(o, lse, *_oracle(p), elem="f16")


def test_paged_krows_stress(fa):
    p = I.make_paged(4, 8, 2, 2, [3000, 2049, 777, 8191], 128, causal=True, seed=33, k_row_frac=0.01)
    o, lse = _run(fa, p)
    compare(o, lse, *_oracle(p))


def test_paged_matches_contiguous_forward(fa):
    # every sequence as long as the cache: same kernel, same plan as fa_forward
    # over the keys stored contiguously, so the outputs are bit-identical
    import torch
    B, Hq, Hkv, Nq, d = 4, 8, 2, 2, 128
    L = 24 * 128
    p = I.make_paged(B, Hq, Hkv, Nq, [L] * B, d, causal=True, seed=34)
    a = I.make_inputs(B, Hq, Hkv, Nq, L, d, causal=True, seed=34)
    o_p, l_p = _run(fa, p)
    o_c, l_c = fa.fa_forward(to_dev(a.q), to_dev(a.k), to_dev(a.v), causal=True, scale=a.scale)
    torch.cuda.synchronize()
    assert np.array_equal(o_p, o_c.float().cpu().numpy().astype(np.float64))
    assert np.array_equal(l_p, l_c.cpu().numpy().astype(np.float64))


def test_paged_decode_workload_full_size(fa):
    # the decode workload (batch 16, 32 query / 8 KV heads, 8192 keys, d = 128)
    # with its cache in shuffled pages: every output against the oracle
    p = I.make_paged(16, 32, 8, 1, [8192] * 16, 128, seed=0)
    o, lse = _run(fa, p)
    compare(o, lse, *_oracle(p))
