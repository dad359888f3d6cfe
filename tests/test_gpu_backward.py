"""GPU parity of libfa's attention backward (fa_backward through the C ABI)
against the FP64 oracle's gradients, element by element, on seeded inputs.

The forward's O and LSE that the backward consumes come from the oracle (O
rounded to the tensors' 16-bit type, LSE to FP32), so the only arithmetic under
test is the backward's own.

Tolerance, derived from the precision the kernels compute in (unit roundoff
u = 2^-8 for BF16, 2^-11 for FP16; scores, sums and accumulators in FP32):
  * P is rounded to 16 bits before dV = P^T dO, dS before dQ = scale dS K and
    dK = scale dS^T Q, and O enters D = rowsum(dO * O) already rounded; the
    oracle's ``backward_error_terms`` evaluates each of those first-order
    effects on absolute values;
  * the gradients themselves are rounded to 16 bits (u |gradient|).
Every element must satisfy |err| <= u (terms + |gradient|); FP32 rounding of the
accumulations is orders of magnitude below that. The relative L2 error is also
bounded (1e-2 BF16, 2e-3 FP16)."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096
FILL = -12345.0


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


def _guarded(torch, shape, dtype):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), FILL, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


def _intact(buf):
    import torch
    n = buf.numel() - 2 * GUARD
    ref = torch.full((GUARD,), FILL, dtype=buf.dtype, device=buf.device)
    return bool(torch.equal(buf[:GUARD], ref)) and bool(torch.equal(buf[GUARD + n:], ref))


def _forward_inputs(a):
    """The oracle's O (rounded to the inputs' 16-bit type) and LSE (FP32)."""
    o, lse = oracle.attention_reference(a.q, a.k, a.v, causal=a.causal, scale=a.scale)
    o16 = I.f64_to_f16(o) if a.dtype == "f16" else I.f64_to_bf16_bits(o)
    return o16, lse.astype(np.float32)


def _run_backward(fa, a, do, o16, lse32):
    """fa_backward with dq, dk, dv inside canary margins that must stay untouched."""
    import torch
    q, k, v, o, dod = to_dev(a.q), to_dev(a.k), to_dev(a.v), to_dev(o16), to_dev(do)
    lse = torch.from_numpy(np.ascontiguousarray(lse32)).cuda()
    dt = q.dtype
    bq, dq = _guarded(torch, tuple(q.shape), dt)
    bk, dk = _guarded(torch, tuple(k.shape), dt)
    bv, dv = _guarded(torch, tuple(v.shape), dt)
    r = fa.fa_backward(q, k, v, o, lse, dod, causal=a.causal, scale=a.scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert r[0].data_ptr() == dq.data_ptr() and r[1].data_ptr() == dk.data_ptr()
    assert r[2].data_ptr() == dv.data_ptr()
    assert _intact(bq) and _intact(bk) and _intact(bv)
    return [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]


def check_gradients(a, do, got, rel_tol=None):
    refs = oracle.attention_backward(a.q, a.k, a.v, do, causal=a.causal, scale=a.scale)
    terms = oracle.backward_error_terms(a.q, a.k, a.v, do, causal=a.causal, scale=a.scale)
    u = 2.0 ** -11 if a.dtype == "f16" else 2.0 ** -8
    if rel_tol is None:
        rel_tol = 2e-3 if a.dtype == "f16" else 1e-2
    res = {}
    for name, g, r, t in zip(("dq", "dk", "dv"), got, refs, terms):
        assert g.shape == r.shape, name
        assert np.isfinite(g).all(), f"non-finite values in {name}"
        err = np.abs(g - r)
        bound = u * (t + np.abs(r))
        # where the bound is 0 the gradient is exactly 0 (no key seen, or dO = 0)
        worst = float(np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0)).max()) \
            if err.size else 0.0
        nr = float(np.linalg.norm(r))
        rel = float(np.linalg.norm(g - r) / nr) if nr > 0 else float(np.linalg.norm(g))
        res[name] = (worst, rel)
        assert worst <= 1.0, (name, res)
        assert rel <= rel_tol, (name, res)
    return res


SHAPES = [
    # (B, H_q, H_kv, N_q, N_k, d, causal)
    (1, 1, 1, 256, 256, 64, False),
    (1, 1, 1, 1, 1, 64, False),
    (1, 1, 1, 17, 17, 128, True),
    (1, 1, 1, 128, 128, 128, True),
    (1, 2, 1, 300, 700, 128, True),      # GQA, N_q < N_k, ragged tiles on both sides
    (2, 4, 2, 513, 513, 128, True),
    (1, 2, 2, 600, 200, 64, True),       # N_q > N_k: the first rows see no key
    (1, 1, 1, 1000, 1000, 128, False),
    (1, 2, 2, 129, 1000, 128, False),
    (2, 8, 2, 4, 777, 128, True),        # few queries, many keys
    (1, 4, 1, 1536, 1536, 128, True),    # GQA 4, several key blocks per query tile
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:6])) + ("c" if s[6] else ""))
def test_backward_parity(fa, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=7)
    do = I.grad_output(a, seed=7)
    got = _run_backward(fa, a, do, *_forward_inputs(a))
    check_gradients(a, do, got)


FP16 = [
    (1, 2, 1, 300, 700, 128, True),
    (2, 4, 2, 513, 513, 64, False),
    (1, 2, 2, 600, 200, 128, True),
]


@pytest.mark.parametrize("shape", FP16, ids=lambda s: "x".join(map(str, s[:6])) + ("c" if s[6] else ""))
def test_backward_parity_fp16(fa, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=8, dtype="f16")
    do = I.grad_output(a, seed=8)
    got = _run_backward(fa, a, do, *_forward_inputs(a))
    check_gradients(a, do, got)


def test_backward_krows_stress(fa):
    # 1 % of K rows scaled by 8: large, peaked scores, recomputed from LSE alone
    a = I.make_inputs(1, 2, 1, 1024, 1024, 128, causal=True, seed=3, k_row_frac=0.01)
    do = I.grad_output(a, seed=3)
    got = _run_backward(fa, a, do, *_forward_inputs(a))
    check_gradients(a, do, got)


def test_backward_after_gpu_forward(fa):
    # O and LSE from libfa's own forward: the chain a user runs. O now carries
    # the forward's rounding too, so only the relative L2 error is bounded here.
    import torch
    a = I.make_inputs(1, 4, 2, 700, 900, 128, causal=True, seed=12)
    do = I.grad_output(a, seed=12)
    q, k, v, dod = to_dev(a.q), to_dev(a.k), to_dev(a.v), to_dev(do)
    o, lse = fa.fa_forward(q, k, v, causal=True, scale=a.scale)
    dq, dk, dv = fa.fa_backward(q, k, v, o, lse, dod, causal=True, scale=a.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    refs = oracle.attention_backward(a.q, a.k, a.v, do, causal=True, scale=a.scale)
    for g, r in zip((dq, dk, dv), refs):
        g = g.float().cpu().numpy().astype(np.float64)
        assert np.linalg.norm(g - r) / np.linalg.norm(r) <= 1e-2


def test_backward_deterministic(fa):
    a = I.make_inputs(1, 4, 2, 700, 900, 128, causal=True, seed=13)
    do = I.grad_output(a, seed=13)
    fwd = _forward_inputs(a)
    g1 = _run_backward(fa, a, do, *fwd)
    g2 = _run_backward(fa, a, do, *fwd)
    for x, y in zip(g1, g2):
        assert np.array_equal(x, y)


def test_backward_empty(fa):
    import torch
    q = torch.randn(1, 2, 5, 128, device="cuda").bfloat16()
    k = torch.empty(1, 1, 0, 128, device="cuda", dtype=torch.bfloat16)
    o = torch.zeros_like(q)
    lse = torch.full((1, 2, 5), float("-inf"), device="cuda")
    dq = torch.full_like(q, 7.0)
    dq, dk, dv = fa.fa_backward(q, k, k, o, lse, q.clone(), dq=dq)
    torch.cuda.synchronize()
    assert torch.all(dq == 0) and dk.numel() == 0 and dv.numel() == 0


FULL = ["one_head_n8192_d128", "h32_n4096_d128", "h32_n4096_d128_causal", "h32_n16384_d128_causal_krows"]


@pytest.mark.parametrize("name", FULL)
def test_backward_full_size(fa, name):
    # The workloads `bench.py --pass backward` times, whole, in the same launch
    # configuration. Heads are independent, so the sampled KV heads (first and
    # last; the last only past N = 8192, where one FP64 head is ~10 GB of
    # scores) and their query heads take O and LSE from the oracle and are
    # checked element by element; the other heads take them from libfa's forward.
    import torch
    a = I.make_workload(name)
    do = I.grad_output(a, seed=0)
    q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    o, lse = fa.fa_forward(q, k, v, causal=a.causal, scale=a.scale)
    g = a.H_q // a.H_kv
    subs = []
    for hk in ([a.H_kv - 1] if a.N_q > 8192 else sorted({0, a.H_kv - 1})):
        hs = slice(hk * g, (hk + 1) * g)
        sub = I.AttentionInputs(a.q[:, hs], a.k[:, hk:hk + 1], a.v[:, hk:hk + 1], a.B, g, 1, a.N_q, a.N_k,
                                a.d, a.causal, a.scale, a.dtype)
        o16, lse32 = _forward_inputs(sub)
        o[:, hs] = to_dev(o16)
        lse[:, hs] = torch.from_numpy(np.ascontiguousarray(lse32)).cuda()
        subs.append((hk, hs, sub))
    torch.cuda.synchronize()
    dq, dk, dv = fa.fa_backward(q, k, v, o, lse, to_dev(do), causal=a.causal, scale=a.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    for hk, hs, sub in subs:
        got = [dq[:, hs].float().cpu().numpy().astype(np.float64),
               dk[:, hk:hk + 1].float().cpu().numpy().astype(np.float64),
               dv[:, hk:hk + 1].float().cpu().numpy().astype(np.float64)]
        check_gradients(sub, do[:, hs], got)
