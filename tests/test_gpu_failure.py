"""Failure detection without a GPU fault: a bounded wait that runs out is reported
through the device status word and the context stays usable; a failed workspace
allocation is reported before anything is enqueued."""
import ctypes
import time

import numpy as np
import pytest

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


def test_wait_timeout_is_reported_and_context_survives(fa):
    import torch
    lib = fa.lib()
    assert lib.fa_device_status(1) == fa.FA_OK
    t0 = time.perf_counter()
    assert lib.fa_selftest_wait_timeout(5_000_000, None) == fa.FA_OK   # a 5 ms limit
    assert lib.fa_device_status(1) == fa.FA_ERR_TIMEOUT                # synchronises, reads, clears
    assert time.perf_counter() - t0 < 2.0
    assert lib.fa_device_status(1) == fa.FA_OK
    # the context is still usable: an ordinary call matches the oracle
    a = I.make_inputs(1, 2, 1, 300, 500, 128, causal=True, seed=4)
    o, lse = fa.fa_forward(to_dev(a.q), to_dev(a.k), to_dev(a.v), causal=True, scale=a.scale)
    torch.cuda.synchronize()
    assert lib.fa_device_status(1) == fa.FA_OK
    compare(bf16_dev_to_f64(o), lse.cpu().numpy().astype(np.float64), *run_oracle(a))


def test_workspace_failure_is_reported_before_launch(fa, monkeypatch):
    import torch
    monkeypatch.setenv("FA_CLUSTER_MERGE", "0")         # split partials through the workspace
    a = I.make_inputs(1, 1, 1, 8192, 8192, 128, seed=2)
    assert fa.fa_forward_plan(1, 1, 1, 8192, 8192, 128, False)["workspace_bytes"] > 0
    q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    o = torch.full((1, 1, 8192, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 1, 8192), float("nan"), dtype=torch.float32, device="cuda")
    monkeypatch.setenv("FA_TEST_WORKSPACE_FAIL", "1")
    st = fa.lib().fa_forward(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                             ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                             ctypes.c_void_p(lse.data_ptr()), 1, 1, 1, 8192, 8192, 128, 0,
                             ctypes.c_float(a.scale), None)
    assert st == fa.FA_ERR_NO_MEMORY
    torch.cuda.synchronize()
    assert bool(torch.isnan(o.float()).all()) and bool(torch.isnan(lse).all())   # nothing ran
    monkeypatch.setenv("FA_TEST_WORKSPACE_FAIL", "0")
    o2, lse2 = fa.fa_forward(q, k, v, causal=False, scale=a.scale)
    torch.cuda.synchronize()
    assert fa.lib().fa_device_status(1) == fa.FA_OK
