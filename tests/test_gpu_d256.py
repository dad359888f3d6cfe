"""GPU parity of the head-dimension-256 forward (fa_forward / fa_forward_fp16
with d = 256: one 128-row query tile per CTA, two score buffers in turn)
against the FP64 oracle, element by element under the same bounds as the other
head dimensions: ragged lengths, causal masks (square, N_q < N_k, N_q > N_k with
rows that see no key), GQA, rows on scaled keys, both element types, and the
32-head N = 4096 workload at full size."""
import numpy as np
import pytest

from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import bf16_dev_to_f64, compare, run_oracle, to_dev

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
    """Forward with O and LSE inside canary margins that must stay untouched."""
    import torch
    q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    B, H_q, H_kv, N_q, N_k, d = a.shape_args
    odt = torch.float16 if a.dtype == "f16" else torch.bfloat16
    n_o, n_l = B * H_q * N_q * d, B * H_q * N_q
    ob = torch.full((n_o + 2 * GUARD,), -12345.0, dtype=odt, device="cuda")
    lb = torch.full((n_l + 2 * GUARD,), -12345.0, dtype=torch.float32, device="cuda")
    o = ob[GUARD:GUARD + n_o].view(B, H_q, N_q, d)
    lse = lb[GUARD:GUARD + n_l].view(B, H_q, N_q)
    fa.fa_forward(q, k, v, causal=a.causal, scale=a.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    for buf, n in ((ob, n_o), (lb, n_l)):
        assert bool(torch.all(buf[:GUARD] == -12345.0)) and bool(torch.all(buf[GUARD + n:] == -12345.0))
    return bf16_dev_to_f64(o), lse.cpu().numpy().astype(np.float64)


SHAPES = [
    # (B, H_q, H_kv, N_q, N_k, causal, k_row_frac, scale)
    (1, 1, 1, 1, 1, False, 0.0, None),
    (1, 1, 1, 17, 17, True, 0.0, None),
    (1, 1, 1, 128, 128, False, 0.0, None),
    (1, 1, 1, 129, 129, True, 0.0, None),
    (1, 2, 1, 255, 255, True, 0.01, None),
    (1, 1, 1, 256, 256, False, 0.0, None),
    (2, 8, 2, 300, 700, True, 0.01, None),     # GQA, N_q < N_k
    (2, 8, 2, 300, 700, False, 0.0, None),
    (1, 4, 4, 600, 200, True, 0.0, None),      # N_q > N_k: leading rows see no key
    (3, 4, 1, 64, 1000, False, 0.0, None),     # GQA group 4, one partial query tile
    (2, 4, 2, 1, 777, True, 0.0, None),        # one query row per head (decode-shaped)
    (1, 2, 2, 512, 4096, False, 0.0, 0.1),     # larger scale: many rescales of O
    (1, 3, 3, 1000, 1000, True, 0.02, None),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + ("c" if s[5] else ""))
def test_d256_shapes(fa, shape, dtype):
    B, Hq, Hkv, Nq, Nk, causal, frac, scale = shape
    a = I.make_inputs(B, Hq, Hkv, Nq, Nk, 256, causal=causal, seed=41, k_row_frac=frac, scale=scale,
                      dtype=dtype)
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a), elem=dtype)


@pytest.mark.parametrize("name", ["h32_n4096_d256", "h32_n4096_d256_causal"])
def test_d256_h32_n4096(fa, name):
    a = I.make_workload(name)
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))


def test_d256_deterministic_and_noalloc(fa):
    # same kernel through fa_forward_noalloc (no scratch at d = 256): same bits
    import torch
    a = I.make_inputs(1, 2, 1, 700, 900, 256, causal=True, seed=42, k_row_frac=0.01)
    o1, l1 = _run(fa, a)
    o2, l2 = _run(fa, a)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    o3, l3 = fa.fa_forward_noalloc(to_dev(a.q), to_dev(a.k), to_dev(a.v), causal=True, scale=a.scale)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_dev_to_f64(o3), o1)
    assert np.array_equal(l3.cpu().numpy().astype(np.float64), l1)


@pytest.mark.parametrize("group", [None, "1", "3"], ids=["default", "g1", "g3"])
def test_d256_causal_head_groups(fa, group, monkeypatch):
    # causal tiles run longest first across groups of heads; groups of 3 leave a
    # short last group, and every tile must still be written exactly once
    if group is None:
        monkeypatch.delenv("FA_CAUSAL_HEAD_GROUP", raising=False)
    else:
        monkeypatch.setenv("FA_CAUSAL_HEAD_GROUP", group)
    a = I.make_inputs(2, 10, 5, 700, 900, 256, causal=True, seed=43, k_row_frac=0.01)
    o, lse = _run(fa, a)
    compare(o, lse, *run_oracle(a))
