"""GPU parity: libfa's fused forward (through the C ABI) against the FP64 oracle,
element by element, on seeded inputs; plus edge cases and determinism."""
import math

import numpy as np
import pytest

import oracle
from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import compare, to_dev, bf16_dev_to_f64, run_oracle

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


GUARD = 4096   # elements of canary before and after O and LSE (16-byte multiples)


def _guarded(torch, shape, dtype, fill):
    """A tensor of `shape` inside a larger buffer whose margins hold `fill`."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


def _margins_intact(buf, fill):
    import torch
    n = buf.numel() - 2 * GUARD
    ref = torch.full((GUARD,), fill, dtype=buf.dtype, device=buf.device)
    return bool(torch.equal(buf[:GUARD], ref)) and bool(torch.equal(buf[GUARD + n:], ref))


def _run(fa, a, naive=False):
    """Run through the binding with O and LSE inside canary margins; the margins
    must be untouched afterwards (no write outside the outputs)."""
    import torch
    q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    B, H_q, H_kv, N_q, N_k, d = a.shape_args
    odt = torch.float16 if a.dtype == "f16" else torch.bfloat16
    ob, o = _guarded(torch, (B, H_q, N_q, d), odt, -12345.0)
    lb, lse = _guarded(torch, (B, H_q, N_q), torch.float32, -12345.0)
    fn = fa.fa_naive_forward if naive else fa.fa_forward
    o2, lse2 = fn(q, k, v, causal=a.causal, scale=a.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert o2.data_ptr() == o.data_ptr() and lse2.data_ptr() == lse.data_ptr()
    assert _margins_intact(ob, -12345.0) and _margins_intact(lb, -12345.0)
    return bf16_dev_to_f64(o), lse.cpu().numpy().astype(np.float64)


SMALL = [
    # (B, H_q, H_kv, N_q, N_k, d, causal)
    (1, 1, 1, 1, 1, 64, False),
    (1, 1, 1, 17, 17, 128, True),
    (1, 1, 1, 127, 127, 64, False),
    (1, 1, 1, 128, 128, 128, True),
    (1, 1, 1, 129, 129, 128, False),
    (1, 2, 1, 255, 255, 64, True),
    (1, 1, 1, 256, 256, 128, True),
    (1, 1, 1, 257, 257, 128, True),
    (2, 2, 2, 383, 383, 64, True),
    (1, 3, 3, 513, 513, 128, False),
    (2, 8, 2, 300, 700, 128, True),     # GQA, N_q < N_k
    (2, 8, 2, 300, 700, 128, False),
    (1, 4, 4, 600, 200, 64, True),      # N_q > N_k: leading rows see no key
    (1, 2, 1, 1000, 1000, 128, False),
    (3, 4, 1, 64, 1000, 128, False),    # GQA group 4
    (1, 1, 1, 1, 5000, 128, False),     # one query row, long key range
    # decode path: G * N_q <= 16 rows per KV head
    (2, 8, 2, 4, 777, 128, True),       # GQA 4 x 4 queries = 16 rows, ragged chunk
    (1, 16, 1, 1, 300, 64, False),      # MQA, 16 heads on one KV head
    (2, 4, 4, 3, 130, 128, True),       # 3 queries, causal, just past one chunk
    (1, 2, 2, 16, 16, 64, True),        # square causal inside one chunk
    (1, 2, 1, 8, 5, 128, True),         # N_q > N_k: leading rows see no key
    (3, 8, 8, 1, 128, 128, False),      # exactly one chunk
    # decode CTAs that walk runs of chunks (128 KV heads: 2 runs of 17 and 16 chunks per head)
    (8, 32, 16, 4, 4100, 128, True),    # GQA 2 x 4 queries, causal
    (16, 8, 8, 1, 4200, 64, False),     # MQA-free, d = 64
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:6])) + ("c" if s[6] else ""))
def test_small_shapes(fa, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=1)
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))


# Split plans: every query block's key range is cut over several CTAs. The
# partials are merged either inside a thread-block cluster (default when every
# block is split) or by the merge kernel (FA_CLUSTER_MERGE=0); both against the oracle.
SPLIT = [
    (1, 1, 1, 8192, 8192, 128, False),   # 32 blocks x 4 key ranges (the one-head workload)
    (1, 1, 1, 2000, 3000, 64, False),    # ragged, d = 64, eight key ranges
    (2, 3, 1, 700, 1500, 128, True),     # causal, GQA, unequal ranges inside a cluster
    (1, 1, 1, 256, 2048, 128, False),    # a single block
    (16, 32, 8, 1, 8192, 128, False),    # decode: runs of chunks per KV head, merged either way
]


@pytest.mark.parametrize("cluster_merge", [True, False], ids=["cluster", "kernel"])
@pytest.mark.parametrize("shape", SPLIT, ids=lambda s: "x".join(map(str, s[:6])) + ("c" if s[6] else ""))
def test_split_merge_modes(fa, shape, cluster_merge, monkeypatch):
    monkeypatch.setenv("FA_CLUSTER_MERGE", "1" if cluster_merge else "0")
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=5, k_row_frac=0.01)
    plan = fa.fa_forward_plan(B, Hq, Hkv, Nq, Nk, d, causal)
    # work units before splitting: 256-row query blocks, or KV heads on the decode
    # path (at most 16 query rows read one KV head)
    blocks = B * Hkv if (Hq // Hkv) * Nq <= 16 else B * Hq * ((Nq + 255) // 256)
    assert plan["ctas"] > blocks                     # the key ranges are split
    if cluster_merge:
        assert plan["launches"] == 1 and plan["workspace_bytes"] == 0
    else:
        assert plan["launches"] == 2 and plan["workspace_bytes"] > 0
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))


CAUSAL_GROUPS = [
    (2, 8, 2, 2560, 2560, 64, True),     # 160 whole blocks (more than a wave), GQA 4
    (1, 10, 5, 2048, 2048, 128, True),   # 80 blocks: split key ranges, merged by block number
    (1, 6, 6, 1500, 3000, 128, True),    # N_q < N_k, ragged last block
]


@pytest.mark.parametrize("group", [None, "1", "3"], ids=["default", "g1", "g3"])
@pytest.mark.parametrize("shape", CAUSAL_GROUPS, ids=lambda s: "x".join(map(str, s[:6])))
def test_causal_head_groups(fa, shape, group, monkeypatch):
    # causal blocks run longest first across groups of heads; groups of 3 leave a
    # short last group, and every block must still be written exactly once
    if group is None:
        monkeypatch.delenv("FA_CAUSAL_HEAD_GROUP", raising=False)
    else:
        monkeypatch.setenv("FA_CAUSAL_HEAD_GROUP", group)
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=9, k_row_frac=0.01)
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))


FP16 = [
    (1, 1, 1, 17, 17, 128, True),
    (1, 2, 1, 255, 255, 64, True),
    (2, 8, 2, 300, 700, 128, True),      # GQA, N_q < N_k
    (1, 4, 4, 600, 200, 64, True),       # N_q > N_k: leading rows see no key
    (1, 1, 1, 2048, 8192, 128, False),   # split key ranges, in-cluster merge
    (2, 8, 2, 2560, 2560, 64, True),     # more than a wave, causal head groups
    (2, 8, 2, 4, 777, 128, True),        # decode path, ragged chunk
    (16, 32, 8, 1, 8192, 128, False),    # decode workload's shape
]


@pytest.mark.parametrize("shape", FP16, ids=lambda s: "x".join(map(str, s[:6])) + ("c" if s[6] else ""))
def test_fp16_parity(fa, shape):
    # FP16 tensors through fa_forward_fp16: same kernels with FP16 operands, P and O
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=21, k_row_frac=0.01, dtype="f16")
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a), elem="f16")


@pytest.mark.parametrize("cluster_merge", [True, False], ids=["cluster", "kernel"])
def test_fp16_split_merge_modes(fa, cluster_merge, monkeypatch):
    monkeypatch.setenv("FA_CLUSTER_MERGE", "1" if cluster_merge else "0")
    a = I.make_inputs(1, 2, 1, 1000, 6000, 128, causal=True, seed=22, dtype="f16")
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a), elem="f16")


def test_fp16_large_scores(fa):
    # scores spread over many octaves: the lazy rescale keeps every FP16 P <= 2^15
    a = I.make_inputs(1, 2, 2, 512, 4096, 128, causal=False, seed=23, scale=0.6, dtype="f16")
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a), elem="f16")


def test_tiny_workload_n256_d64(fa):
    a = I.make_workload("tiny_n256_d64")
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))


def test_one_head_n8192_d128(fa):
    # the split-key path: 32 query blocks are too few for the GPU, so each block's
    # key range is split over several CTAs and merged in-kernel
    a = I.make_workload("one_head_n8192_d128")
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))


@pytest.mark.parametrize("name", ["h32_n4096_d128", "h32_n4096_d128_causal"])
def test_h32_n4096(fa, name):
    a = I.make_workload(name)
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))


def test_decode_b16_h32_kv8(fa):
    a = I.make_workload("decode_b16_h32_kv8_n8192_d128")
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))


DECODE_REGIMES = [
    # (B, H_q, H_kv, N_q, N_k, d, causal), launches: how the decode plan splits each KV head
    ((1, 8, 2, 1, 40000, 128, False), 2),   # 2 KV heads, 313 chunks: runs merged by the merge kernel
    ((4, 32, 8, 1, 6000, 64, False), 1),    # 32 KV heads: 8 parts per head in clusters of 8
    ((8, 16, 8, 2, 3000, 128, True), 1),    # 64 KV heads, 2 query rows each: 4 parts, causal
    ((64, 32, 8, 1, 1000, 128, False), 1),  # 512 KV heads: one part each, no merge
]


@pytest.mark.parametrize("shape,launches", DECODE_REGIMES, ids=lambda s: "x".join(map(str, s[:6])) if isinstance(s, tuple) else None)
def test_decode_plan_regimes(fa, shape, launches):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    assert fa.fa_forward_plan(B, Hq, Hkv, Nq, Nk, d, causal)["launches"] == launches
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=14, k_row_frac=0.01)
    compare(*_run(fa, a), *run_oracle(a))


def test_deterministic(fa):
    a = I.make_inputs(1, 2, 1, 1000, 1500, 128, causal=True, seed=4, k_row_frac=0.01)
    o1, l1 = _run(fa, a)
    o2, l2 = _run(fa, a)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_empty_keys_and_queries(fa):
    import torch
    q = torch.randn(1, 2, 5, 128, device="cuda").bfloat16()
    k = torch.empty(1, 1, 0, 128, device="cuda", dtype=torch.bfloat16)
    o, lse = fa.fa_forward(q, k, k)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    q0 = torch.empty(1, 2, 0, 128, device="cuda", dtype=torch.bfloat16)
    o0, l0 = fa.fa_forward(q0, q, q)
    assert o0.numel() == 0


def naive_lse_bound(a):
    """Per-row LSE tolerance of the unfused path: it stores S in BF16, so each
    score carries a relative rounding error up to u = 2^-8, and
    |dLSE_i| = |sum_j p_ij dS_ij| <= u * max_j |s_ij| <= u * scale * |q_i| * max_j |k_j|."""
    from oracle.attention import bf16_to_f64
    qf, kf = bf16_to_f64(a.q), bf16_to_f64(a.k)
    g = a.H_q // a.H_kv
    kmax = np.repeat(np.linalg.norm(kf, axis=-1).max(-1), g, axis=1)     # [B, H_q]
    return 2.0 ** -8 * a.scale * np.linalg.norm(qf, axis=-1) * kmax[..., None] + 1e-4


def test_naive_matches_oracle(fa):
    # O: BF16 P adds a relative error <= 2^-8 per weight on top of the score rounding;
    # the bound used is twice the fused path's (max|dO| <= 2e-2, rel L2 <= 1e-2).
    for shape in [(1, 1, 1, 256, 256, 64, False), (1, 2, 1, 300, 517, 128, True),
                  (2, 4, 2, 129, 129, 128, False)]:
        a = I.make_inputs(*shape[:6], causal=shape[6], seed=2)
        o, lse = _run(fa, a, naive=True)
        o_ref, lse_ref, a_ref = run_oracle(a)
        compare(o, None, o_ref, None, a_ref, tol_o=2e-2, tol_rel=1e-2)
        bound = naive_lse_bound(a)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isneginf(lse), ~fin)
        assert np.all(np.abs(lse - lse_ref)[fin] <= bound[fin])


def test_naive_one_head_n8192(fa):
    a = I.make_workload("one_head_n8192_d128")
    o, lse = _run(fa, a, naive=True)
    o_ref, lse_ref, a_ref = run_oracle(a)
    compare(o, None, o_ref, None, a_ref, tol_o=2e-2, tol_rel=1e-2)
    assert np.all(np.abs(lse - lse_ref) <= naive_lse_bound(a))


def test_rejects_memory_not_on_the_current_device(fa):
    # every pointer must be memory of the current GPU: pinned host memory (which
    # the GPU could reach) and ordinary host memory are refused before anything
    # is enqueued; the same call with device tensors runs
    import torch
    a = I.make_inputs(1, 2, 1, 200, 300, 128, causal=True, seed=12)
    q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    o = torch.zeros((1, 2, 200, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 200), dtype=torch.float32, device="cuda")
    pinned = q.cpu().pin_memory()
    plain = np.zeros(q.numel() + 64, dtype=np.uint16)
    addr = plain.ctypes.data
    host_ptr = addr + (-addr) % 16          # 16-byte aligned host address
    L = fa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    args = lambda qq, oo: (qq, k.data_ptr(), v.data_ptr(), oo, lse.data_ptr(), 1, 2, 1, 200, 300, 128, 1,
                           a.scale, stream)
    for bad_q in (pinned.data_ptr(), host_ptr):
        assert L.fa_forward(*args(bad_q, o.data_ptr())) == fa.FA_ERR_INVALID_ARG
        assert L.fa_forward_noalloc(*args(bad_q, o.data_ptr())) == fa.FA_ERR_INVALID_ARG
    pinned_o = torch.zeros((1, 2, 200, 128), dtype=torch.bfloat16).pin_memory()
    assert L.fa_forward(*args(q.data_ptr(), pinned_o.data_ptr())) == fa.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(pinned_o == 0)
    assert L.fa_forward(*args(q.data_ptr(), o.data_ptr())) == fa.FA_OK
    torch.cuda.synchronize()
    compare(bf16_dev_to_f64(o), lse.cpu().numpy().astype(np.float64), *run_oracle(a))
    # the backward and the paged decode check their pointers the same way
    dq = torch.empty_like(q)
    st = L.fa_backward(pinned.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       o.data_ptr(), dq.data_ptr(), torch.empty_like(k).data_ptr(),
                       torch.empty_like(v).data_ptr(), 1, 2, 1, 200, 300, 128, 1, a.scale, 0, stream)
    assert st == fa.FA_ERR_INVALID_ARG
