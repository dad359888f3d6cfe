"""Shared helpers for the GPU parity tests (device transfer, tolerance checks)."""
import numpy as np

import oracle

# Tolerances on BF16 inputs (FP32 accumulate, BF16 output)
TOL_MAX_ABS_O = 1e-2
TOL_REL_L2_O = 5e-3
TOL_MAX_ABS_LSE = 1e-3
# Element-wise, the absolute bound on O is widened where the BF16 arithmetic
# the method fixes cannot meet 1e-2: BF16 has unit roundoff u = 2^-8, so
#   * rounding O itself to BF16 moves it by up to u |O|, and
#   * each probability is rounded to BF16 before the PV product, which moves
#     O_t = sum_j p_j v_jt / l by up to u * A_t with A_t = sum_j p_j |v_jt| / l.
# A is the oracle's own definition evaluated on |V|. Each element must satisfy
#   |dO| <= max(1e-2, TOL_REL_ELEM_O * (A + |O_ref|))   (5e-3 = 1.28 u).
TOL_REL_ELEM_O = 5e-3
# The same derivation with FP16's unit roundoff u = 2^-11 (P and O rounded to
# FP16): 1.28 u = 6.25e-4; the absolute floor (1e-2) stays the stated one.
TOL_REL_ELEM_O_F16 = 6.25e-4


def abs_values(v):
    """|V| in V's own storage (FP16 values, or BF16 bit patterns with the sign
    bit cleared); exact either way."""
    v = np.asarray(v)
    if v.dtype == np.float16:
        return np.abs(v)
    return v.astype(np.uint16) & np.uint16(0x7FFF)


def to_dev(x):
    """Input array to a CUDA tensor: FP16 values as torch.float16, BF16 bit
    patterns as torch.bfloat16."""
    import torch
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return torch.from_numpy(x).cuda()
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()


def bf16_dev_to_f64(t):
    import torch
    return t.float().cpu().numpy().astype(np.float64)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, o_abs_ref=None, tol_o=TOL_MAX_ABS_O,
            tol_rel=TOL_REL_L2_O, tol_lse=TOL_MAX_ABS_LSE, elem="bf16"):
    """Element-wise comparison of O and LSE; returns a dict of error figures.
    ``elem`` ("bf16" or "f16") picks the element-wise relative bound."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape
    assert np.isfinite(o_gpu).all(), "non-finite values in O"
    err = np.abs(o_gpu - o_ref)
    max_abs = float(err.max()) if err.size else 0.0
    a_ref = np.abs(o_ref) if o_abs_ref is None else np.asarray(o_abs_ref, dtype=np.float64)
    rel_elem = TOL_REL_ELEM_O_F16 if elem == "f16" else TOL_REL_ELEM_O
    bound = np.maximum(tol_o, rel_elem * (a_ref + np.abs(o_ref)))
    worst = float((err / bound).max()) if err.size else 0.0
    denom = float(np.linalg.norm(o_ref))
    rel = float(np.linalg.norm(o_gpu - o_ref) / denom) if denom > 0 else float(np.linalg.norm(o_gpu))
    res = {"max_abs_o": max_abs, "rel_l2_o": rel, "worst_over_bound": worst}
    if lse_ref is not None:
        lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse_gpu), inf_ref), "LSE -inf pattern differs"
        fin = ~inf_ref
        lerr = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
        res["max_abs_lse"] = lerr
        assert lerr <= tol_lse, res
    assert worst <= 1.0, res
    assert rel <= tol_rel, res
    return res


def run_oracle(a):
    """(O, LSE, A): the oracle's O and LSE, and A = the same attention of |V|."""
    o, lse = oracle.attention_reference(a.q, a.k, a.v, causal=a.causal, scale=a.scale)
    o_abs, _ = oracle.attention_reference(a.q, a.k, abs_values(a.v), causal=a.causal, scale=a.scale)
    return o, lse, o_abs
