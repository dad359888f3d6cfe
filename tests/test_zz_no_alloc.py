"""fa_forward_noalloc: the entry point for callers that cannot allocate device
memory (for example a serving loop that must never block in cudaMalloc, or a
process whose device memory is all reserved up front by another allocator).
It must give the same results as fa_forward, whose split partials come from a
pool allocation, while using only libfa's fixed scratch array.

This file is named to be collected last, so a failure here comes after every
other test has run. It passes alone in a fresh process and after the others.
"""
import ctypes
import math

import numpy as np
import pytest

from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import compare, run_oracle, to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


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


def _call(fa, entry, q, k, v, o, lse, a):
    """Call an entry point through the C ABI with raw device pointers."""
    import torch
    f = getattr(fa.lib(), entry)
    st = f(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
           ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
           ctypes.c_void_p(lse.data_ptr()), a.B, a.H_q, a.H_kv, a.N_q, a.N_k, a.d, int(a.causal),
           ctypes.c_float(a.scale), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _planned_scratch(fa, a):
    """Scratch bytes of the split partials (the library's own plan for this request)."""
    return fa.fa_forward_plan(a.B, a.H_q, a.H_kv, a.N_q, a.N_k, a.d, a.causal)["workspace_bytes"]


@pytest.mark.parametrize("shape,cluster_merge", [
    # split partials through the scratch array (merge kernel)
    ((1, 1, 1, 8192, 8192, 128, False), False),   # one head, N = 8192: split over 4 CTAs per block
    ((1, 2, 1, 700, 3000, 64, True), False),      # causal, GQA, ragged, d = 64
    # decode partials through the scratch array (chunk-merge kernel)
    ((2, 8, 2, 1, 4096, 128, False), False),      # GQA 4, one query row: runs of 128-key chunks
    # split partials merged inside clusters: no scratch at all
    ((1, 1, 1, 8192, 8192, 128, False), True),
])
def test_noalloc_matches_fa_forward_twice(fa, shape, cluster_merge, monkeypatch):
    import torch
    monkeypatch.setenv("FA_CLUSTER_MERGE", "1" if cluster_merge else "0")
    a = I.make_inputs(*shape[:6], causal=shape[6], seed=3, k_row_frac=0.01)
    q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    if cluster_merge:
        assert _planned_scratch(fa, a) == 0
    else:
        assert 0 < _planned_scratch(fa, a) <= SCRATCH_BYTES   # the scratch path is exercised
    o_ref = torch.empty((a.B, a.H_q, a.N_q, a.d), dtype=torch.bfloat16, device="cuda")
    l_ref = torch.empty((a.B, a.H_q, a.N_q), dtype=torch.float32, device="cuda")
    assert _call(fa, "fa_forward", q, k, v, o_ref, l_ref, a) == fa.FA_OK
    torch.cuda.synchronize()
    ref_o = o_ref.float().cpu().numpy()
    ref_l = l_ref.cpu().numpy()
    oracle_o, oracle_l, oracle_a = run_oracle(a)
    for _ in range(2):   # two calls in a row: the array keeps the previous call's contents
        o = torch.full_like(o_ref, float("nan"))
        l = torch.full_like(l_ref, float("nan"))
        assert _call(fa, "fa_forward_noalloc", q, k, v, o, l, a) == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.fa_device_status() == fa.FA_OK
        got_o = o.float().cpu().numpy()
        got_l = l.cpu().numpy()
        # the same kernels and the same split as fa_forward: the same bits
        assert np.array_equal(got_o, ref_o)
        assert np.array_equal(got_l, ref_l)
        # and within the method's tolerances of the FP64 oracle
        compare(got_o.astype(np.float64), got_l.astype(np.float64), oracle_o, oracle_l, oracle_a)


def test_noalloc_rejects_requests_beyond_scratch(fa, monkeypatch):
    import torch
    monkeypatch.setenv("FA_CLUSTER_MERGE", "0")   # partials through the scratch array
    # find a shape whose planned split partials exceed the fixed array
    for heads in range(40, 160, 4):
        a = I.make_inputs(1, heads, heads, 256, 4096, 128, seed=0)
        if _planned_scratch(fa, a) > SCRATCH_BYTES:
            break
    else:
        pytest.skip("no candidate shape exceeds the scratch on this GPU")
    q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    o = torch.zeros((a.B, a.H_q, a.N_q, a.d), dtype=torch.bfloat16, device="cuda")
    l = torch.zeros((a.B, a.H_q, a.N_q), dtype=torch.float32, device="cuda")
    assert _call(fa, "fa_forward_noalloc", q, k, v, o, l, a) == fa.FA_ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert torch.all(o == 0)   # nothing was enqueued
    # the same request through fa_forward (pool-allocated partials) is fine
    assert _call(fa, "fa_forward", q, k, v, o, l, a) == fa.FA_OK
