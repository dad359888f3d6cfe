"""The FA_DEBUG build of libfa (device-side bounds checks that record a status
code and skip the access, the stand-in for a memory checker): it builds, its
self-test reports FA_ERR_BOUNDS through the status word, and the small and
ragged shapes, split plans (both merge routes), decode shapes, d = 256, FP8
inputs and the backward all run under it with no bounds report and results
within the oracle's tolerances."""
import ctypes

import numpy as np
import pytest

from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import TOL_REL_L2_O_FP8, compare, run_oracle, run_oracle_fp8, to_dev
from test_gpu_forward import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import exact_tiled_attention_forward_gb300 as fa
    from exact_tiled_attention_forward_gb300 import build
    path = build.build(debug=True)
    lib = ctypes.CDLL(path)
    for name, (res, args) in fa._SIGNATURES.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    assert lib.fa_debug_build() == 1
    build.build()
    assert fa.lib().fa_debug_build() == 0     # the default library has no checks
    return lib


def _status(lib):
    return lib.fa_device_status(1)


def _forward(lib, a, fp8=False):
    import torch
    B, H_q, H_kv, N_q, N_k, d = a.shape_args
    if fp8:
        q, k, v = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (a.q, a.k, a.v))
    else:
        q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    odt = torch.float16 if a.dtype == "f16" else torch.bfloat16
    o = torch.empty((B, H_q, N_q, d), dtype=odt, device="cuda")
    lse = torch.empty((B, H_q, N_q), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H_q, H_kv, N_q,
            N_k, d, int(a.causal), a.scale)
    if fp8:
        st = lib.fa_forward_fp8(*args, *a.descale, stream)
    elif a.dtype == "f16":
        st = lib.fa_forward_fp16(*args, stream)
    else:
        st = lib.fa_forward(*args, stream)
    assert st == 0
    torch.cuda.synchronize()
    assert _status(lib) == 0, "a bounds check failed"
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def test_bounds_selftest_reports_through_the_status_word(dbg):
    import torch
    assert dbg.fa_selftest_bounds(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    assert _status(dbg) == -7          # FA_ERR_BOUNDS, then cleared
    assert _status(dbg) == 0


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:6])) + ("c" if s[6] else ""))
def test_small_shapes_under_bounds_checks(dbg, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=1)
    compare(*_forward(dbg, a), *run_oracle(a))


@pytest.mark.parametrize("cluster_merge", [True, False], ids=["cluster", "kernel"])
@pytest.mark.parametrize("shape", [(1, 1, 1, 2000, 3000, 64, False), (2, 3, 1, 700, 1500, 128, True),
                                   (16, 32, 8, 1, 8192, 128, False)],
                         ids=["ragged_d64", "causal_gqa", "decode"])
def test_split_plans_under_bounds_checks(dbg, shape, cluster_merge, monkeypatch):
    monkeypatch.setenv("FA_CLUSTER_MERGE", "1" if cluster_merge else "0")
    a = I.make_inputs(*shape[:6], causal=shape[6], seed=5, k_row_frac=0.01)
    compare(*_forward(dbg, a), *run_oracle(a))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_d256_under_bounds_checks(dbg, dtype):
    a = I.make_inputs(2, 8, 2, 300, 700, 256, causal=True, seed=6, k_row_frac=0.01, dtype=dtype)
    compare(*_forward(dbg, a), *run_oracle(a), elem=dtype)


def test_fp8_under_bounds_checks(dbg):
    a = I.make_inputs(2, 8, 2, 300, 700, 128, causal=True, seed=7, k_row_frac=0.01, dtype="e4m3")
    o, lse = _forward(dbg, a, fp8=True)
    o_ref, lse_ref, a_ref, e_ref = run_oracle_fp8(a)
    compare(o, lse, o_ref, lse_ref, a_ref, tol_rel=TOL_REL_L2_O_FP8, elem="e4m3", fp8_e=e_ref)


@pytest.mark.parametrize("shape", [(1, 1, 1, 17, 17, 128, True, "bf16"), (1, 2, 1, 300, 700, 128, True, "bf16"),
                                   (1, 2, 2, 600, 200, 64, True, "bf16"), (2, 4, 2, 513, 513, 64, False, "f16")],
                         ids=["tiny_causal", "gqa_ragged", "nq_gt_nk_d64", "f16_d64"])
def test_backward_under_bounds_checks(dbg, shape):
    import torch
    import test_gpu_backward as TB
    from exact_tiled_attention_forward_gb300 import FA_DTYPE_BF16, FA_DTYPE_FP16
    B, H_q, H_kv, N_q, N_k, d, causal, dtype = shape
    a = I.make_inputs(B, H_q, H_kv, N_q, N_k, d, causal=causal, seed=9, dtype=dtype)
    do = I.grad_output(a, seed=9)
    o16, lse32 = TB._forward_inputs(a)
    q, k, v, o, dod = to_dev(a.q), to_dev(a.k), to_dev(a.v), to_dev(o16), to_dev(do)
    lse = torch.from_numpy(np.ascontiguousarray(lse32)).cuda()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = dbg.fa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dod.data_ptr(),
                         dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H_q, H_kv, N_q, N_k, d, int(causal),
                         a.scale, FA_DTYPE_FP16 if dtype == "f16" else FA_DTYPE_BF16,
                         torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert _status(dbg) == 0, "a bounds check failed"
    got = [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    TB.check_gradients(a, do, got)
