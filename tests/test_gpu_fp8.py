"""GPU parity of fa_forward_fp8 (FP8 E4M3 inputs with per-tensor factors, BF16
output) against the FP64 oracle on the decoded values, element by element,
under the FP8 bound of helpers.py (P rounded to E4M3 before the P V product:
oracle.p_rounding_bound_fp8; O rounded to BF16), relative L2 <= 2^-4 and
|dLSE| <= 1e-3. Shapes: the small and ragged ones, causal and GQA, rows that
see no key, split key ranges merged both ways, rows on scaled keys (running-max
rescales with P kept <= 2^8), and the one-head and 32-head workloads at full
size."""
import numpy as np
import pytest

from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import TOL_REL_L2_O_FP8, compare, run_oracle_fp8

pytestmark = pytest.mark.gpu

GUARD = 4096


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


def _run(fa, a):
    """fa_forward_fp8 with O and LSE inside canary margins that must stay untouched."""
    import torch
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    q, k, v = dev(a.q), dev(a.k), dev(a.v)
    B, H_q, H_kv, N_q, N_k, d = a.shape_args
    n_o, n_l = B * H_q * N_q * d, B * H_q * N_q
    ob = torch.full((n_o + 2 * GUARD,), -12345.0, dtype=torch.bfloat16, device="cuda")
    lb = torch.full((n_l + 2 * GUARD,), -12345.0, dtype=torch.float32, device="cuda")
    o = ob[GUARD:GUARD + n_o].view(B, H_q, N_q, d)
    lse = lb[GUARD:GUARD + n_l].view(B, H_q, N_q)
    fa.fa_forward_fp8(q, k, v, a.descale, causal=a.causal, scale=a.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    for buf, n in ((ob, n_o), (lb, n_l)):
        assert bool(torch.all(buf[:GUARD] == -12345.0)) and bool(torch.all(buf[GUARD + n:] == -12345.0))
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _check(fa, a):
    o, lse = _run(fa, a)
    o_ref, lse_ref, a_ref, e_ref = run_oracle_fp8(a)
    return compare(o, lse, o_ref, lse_ref, a_ref, tol_rel=TOL_REL_L2_O_FP8, elem="e4m3", fp8_e=e_ref)


SMALL = [
    # (B, H_q, H_kv, N_q, N_k, causal, k_row_frac, scale)
    (1, 1, 1, 256, 256, False, 0.0, None),     # the small workload's size
    (1, 1, 1, 1, 1, False, 0.0, None),
    (1, 1, 1, 17, 17, True, 0.0, None),
    (1, 1, 1, 129, 129, False, 0.0, None),
    (1, 2, 1, 255, 255, True, 0.0, None),
    (1, 1, 1, 257, 257, True, 0.01, None),
    (2, 8, 2, 300, 700, True, 0.01, None),     # GQA, N_q < N_k
    (1, 4, 4, 600, 200, True, 0.0, None),      # N_q > N_k: leading rows see no key
    (1, 2, 1, 1000, 1000, False, 0.02, None),
    (3, 4, 1, 64, 1000, False, 0.0, None),     # GQA group 4
    (2, 8, 2, 4, 777, True, 0.0, None),        # decode-shaped: runs the prefill kernel
    (1, 2, 2, 512, 4096, False, 0.0, 0.6),     # large scores: many rescales, P <= 2^8
    (2, 3, 1, 700, 1500, True, 0.01, 0.3),     # causal, GQA, scaled keys, larger scale
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:5])) + ("c" if s[5] else ""))
def test_fp8_small_shapes(fa, shape):
    B, Hq, Hkv, Nq, Nk, causal, frac, scale = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, 128, causal=causal, seed=31, k_row_frac=frac, scale=scale,
                      dtype="e4m3")
    _check(fa, a)


@pytest.mark.parametrize("cluster_merge", [True, False], ids=["cluster", "kernel"])
def test_fp8_split_merge_modes(fa, cluster_merge, monkeypatch):
    # 8 query blocks over 8192 keys: every block's key range split over several CTAs
    monkeypatch.setenv("FA_CLUSTER_MERGE", "1" if cluster_merge else "0")
    a = I.make_inputs(1, 1, 1, 2048, 8192, 128, causal=False, seed=32, k_row_frac=0.01, dtype="e4m3")
    _check(fa, a)


@pytest.mark.parametrize("name", ["one_head_n8192_d128", "h32_n4096_d128", "h32_n4096_d128_causal"])
def test_fp8_workloads(fa, name):
    a = I.make_workload(name, dtype="e4m3")
    res = _check(fa, a)
    assert res["rel_l2_o"] <= TOL_REL_L2_O_FP8


def test_fp8_deterministic(fa):
    a = I.make_inputs(1, 2, 1, 1000, 1500, 128, causal=True, seed=33, k_row_frac=0.01, dtype="e4m3")
    o1, l1 = _run(fa, a)
    o2, l2 = _run(fa, a)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_fp8_rejects_head_dim_256(fa):
    import torch
    q = torch.zeros((1, 1, 64, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError):
        fa.fa_forward_fp8(q, q, q, (1.0, 1.0, 1.0))


# head dimension 64: 64-byte rows, 64-byte swizzled tiles
D64 = [
    (1, 1, 1, 256, 256, False, 0.0),       # the small workload (one head, N = 256, d = 64)
    (1, 1, 1, 17, 17, True, 0.0),
    (1, 2, 1, 255, 255, True, 0.01),
    (2, 8, 2, 300, 700, True, 0.01),       # GQA, N_q < N_k
    (1, 4, 4, 600, 200, True, 0.0),        # rows that see no key
    (1, 1, 1, 2000, 3000, False, 0.0),     # split key ranges
]


@pytest.mark.parametrize("shape", D64, ids=lambda s: "x".join(map(str, s[:5])) + ("c" if s[5] else ""))
def test_fp8_head_dim_64(fa, shape):
    B, Hq, Hkv, Nq, Nk, causal, frac = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, 64, causal=causal, seed=34, k_row_frac=frac, dtype="e4m3")
    _check(fa, a)


def test_fp8_tiny_workload(fa):
    _check(fa, I.make_workload("tiny_n256_d64", dtype="e4m3"))


@pytest.mark.parametrize("cluster_merge", [True, False], ids=["cluster", "kernel"])
def test_fp8_head_dim_64_split_merge_modes(fa, cluster_merge, monkeypatch):
    monkeypatch.setenv("FA_CLUSTER_MERGE", "1" if cluster_merge else "0")
    a = I.make_inputs(1, 1, 1, 2048, 8192, 64, causal=False, seed=35, k_row_frac=0.01, dtype="e4m3")
    _check(fa, a)
