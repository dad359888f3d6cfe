"""The C-ABI library: builds, loads, exports every declared symbol, validates
arguments on the host (no device work is started for a rejected call)."""
import ctypes
import math
import os
import shutil

import pytest

import exact_tiled_attention_forward_gb300 as fa
from exact_tiled_attention_forward_gb300 import build as fa_build

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="CUDA toolkit not installed")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("libfa.so not built and no nvcc")
        fa_build.build()
    return fa.lib()


def test_header_symbols_exported(lib):
    names = fa.header_functions()
    assert set(names) == {"fa_forward", "fa_forward_fp16", "fa_forward_fp8", "fa_forward_host",
                          "fa_forward_host_packed", "fa_debug_build", "fa_selftest_bounds",
                          "fa_backward", "fa_decode_paged",
                          "fa_forward_noalloc",
                          "fa_naive_forward",
                          "fa_naive_workspace_bytes", "fa_forward_plan", "fa_selftest_wait_timeout",
                          "fa_status_string", "fa_get_last_cuda_error", "fa_device_status",
                          "fa_version"}
    for n in names:
        assert hasattr(lib, n), n


def test_single_gpu_library_exports_both_headers(lib):
    # libfa_single_gpu.so = libfa's entry points + the cluster-multicast forward;
    # libfa.so itself has no multicast entry point
    if not os.path.exists(fa.LIB_SINGLE_GPU_PATH):
        fa_build.build()
    single = fa.lib_single_gpu()
    extra = fa.header_functions(fa.HEADER_SINGLE_GPU)
    assert extra == ["fa_forward_cluster_multicast"]
    for n in fa.header_functions() + extra:
        assert hasattr(single, n), n
    assert not hasattr(lib, "fa_forward_cluster_multicast")


def test_default_library_sources_hold_no_multicast():
    # the sources libfa.so is linked from never name a cluster-multicast copy or commit
    for name in os.listdir(fa_build.CSRC):
        text = open(os.path.join(fa_build.CSRC, name)).read()
        assert "multicast::cluster" not in text, name
    assert any("multicast::cluster" in open(os.path.join(fa_build.CSRC_SINGLE, n)).read()
               for n in os.listdir(fa_build.CSRC_SINGLE))


def test_single_gpu_forward_refuses_multi_process_jobs(lib, monkeypatch):
    # checked before anything else: a rank of a multi-process job gets UNSUPPORTED
    if not os.path.exists(fa.LIB_SINGLE_GPU_PATH):
        fa_build.build()
    f = fa.lib_single_gpu().fa_forward_cluster_multicast
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert f(Q, K, V, O, L, 1, 2, 1, 64, 64, 128, 0, 0.125, None) == fa.FA_ERR_UNSUPPORTED
    monkeypatch.setenv("WORLD_SIZE", "1")
    # otherwise it validates like fa_forward
    assert f(Q, K, V, O, L, 1, 3, 2, 64, 64, 128, 0, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert f(Q, K, V, Q, L, 1, 2, 1, 64, 64, 128, 0, 0.125, None) == fa.FA_ERR_INVALID_ARG


def test_debug_build_switch(lib):
    # the default library has no bounds checks and refuses their self-test
    assert lib.fa_debug_build() == 0
    assert lib.fa_selftest_bounds(None) == fa.FA_ERR_UNSUPPORTED


def test_status_strings(lib):
    assert fa.fa_status_string(-7) == "a bounds check of the FA_DEBUG build failed"
    for code in (0, -1, -2, -3, -4, -5, -6, -7, 7):
        s = fa.fa_status_string(code)
        assert isinstance(s, str) and s
    assert fa.fa_status_string(-5) == "kernel wait timed out"
    assert fa.fa_version() == (0, 1)


def test_workspace_bytes(lib):
    assert fa.fa_naive_workspace_bytes(1, 1, 8192, 8192) == 8192 * 8192 * 2
    assert fa.fa_naive_workspace_bytes(2, 3, 5, 9) == 2 * 3 * 5 * 16 * 2   # rows padded to 8
    assert fa.fa_naive_workspace_bytes(-1, 1, 1, 1) == 0


# fake, 16-byte aligned, non-overlapping addresses: validation never dereferences them
Q, K, V, O, L = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def _fwd(lib, q=Q, k=K, v=V, o=O, l=L, B=1, Hq=2, Hkv=1, Nq=64, Nk=64, d=128, causal=0,
         scale=0.125):
    return lib.fa_forward(q, k, v, o, l, B, Hq, Hkv, Nq, Nk, d, causal, scale, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=3, Hkv=2), fa.FA_ERR_INVALID_ARG),            # H_q % H_kv != 0
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=-1), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=-5), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(d=0), fa.FA_ERR_INVALID_ARG),
    (dict(q=0), fa.FA_ERR_INVALID_ARG),                    # null q
    (dict(o=0), fa.FA_ERR_INVALID_ARG),
    (dict(k=0), fa.FA_ERR_INVALID_ARG),
    (dict(q=Q + 8), fa.FA_ERR_INVALID_ARG),                # misaligned
    (dict(l=L + 4), fa.FA_ERR_INVALID_ARG),
    (dict(o=Q + 64), fa.FA_ERR_INVALID_ARG),               # o overlaps q
    (dict(o=V), fa.FA_ERR_INVALID_ARG),                    # o aliases v
    (dict(l=O + 16), fa.FA_ERR_INVALID_ARG),               # lse inside o
    (dict(B=1 << 16, Hq=1 << 8, Hkv=1, Nq=1 << 8), fa.FA_ERR_INVALID_ARG),  # > 2^31 rows
])
def test_forward_rejects(lib, kw, status):
    assert _fwd(lib, **kw) == status


def test_noalloc_rejects_like_forward(lib):
    f = lib.fa_forward_noalloc
    assert f(Q, K, V, O, L, 1, 3, 2, 64, 64, 128, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, 1, 2, 1, 64, 64, 96, 0, 0.1, None) == fa.FA_ERR_UNSUPPORTED
    assert f(Q, K, V, Q, L, 1, 2, 1, 64, 64, 128, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    assert f(0, 0, 0, 0, 0, 1, 2, 1, 0, 64, 128, 0, 0.1, None) == fa.FA_OK


def test_head_dim_256_only_on_the_forward(lib):
    # d = 256 is a forward-only head dimension: the backward, the paged decode and
    # the unfused baseline refuse it before anything else runs
    need = lib.fa_naive_workspace_bytes(1, 2, 64, 64)
    assert lib.fa_naive_forward(Q, K, V, O, L, 1, 2, 1, 64, 64, 256, 0, 0.1, 0x60000000, need,
                                None) == fa.FA_ERR_UNSUPPORTED
    D1, D2, D3 = 0x70000000, 0x80000000, 0x90000000
    assert lib.fa_backward(Q, K, V, O, L, O, D1, D2, D3, 1, 2, 1, 64, 64, 256, 0, 0.1, 0,
                           None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_decode_paged(Q, K, V, D1, D2, O, L, 1, 2, 1, 1, 4, 2, 256, 0, 0.1, 0,
                               None) == fa.FA_ERR_UNSUPPORTED
    plan = fa.fa_forward_plan(2, 4, 2, 300, 500, 256, True)
    assert plan == {"ctas": 2 * 4 * 3, "launches": 1, "workspace_bytes": 0}


def _gpu_present():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def test_fp8_rejects(lib):
    def f(q=Q, k=K, v=V, o=O, l=L, Hq=2, Hkv=1, Nq=64, d=128, scale=0.1, ds=(1.0, 1.0, 1.0)):
        return lib.fa_forward_fp8(q, k, v, o, l, 1, Hq, Hkv, Nq, 64, d, 0, scale, *ds, None)
    assert f(Hq=3, Hkv=2) == fa.FA_ERR_INVALID_ARG                       # H_q % H_kv
    assert f(d=256) == fa.FA_ERR_UNSUPPORTED                              # FP8: d = 64 or 128
    for bad in ((0.0, 1.0, 1.0), (1.0, -1.0, 1.0), (1.0, 1.0, math.inf), (1.0, math.nan, 1.0)):
        assert f(ds=bad) == fa.FA_ERR_INVALID_ARG                         # factors finite, > 0
    assert f(ds=(1e30, 1e30, 1.0)) == fa.FA_ERR_INVALID_ARG                # scale * factors overflows
    # o (BF16, 2 bytes per element) may not overlap q (1 byte per element): q spans
    # 2 * 64 * 128 bytes, so o may start right after it but not inside it
    assert f(o=Q + 64 * 128) == fa.FA_ERR_INVALID_ARG
    if not _gpu_present():   # with a GPU, the made-up pointers then fail the device check
        assert f(o=Q + 2 * 64 * 128) != fa.FA_ERR_INVALID_ARG
    assert f(q=0, k=0, v=0, o=0, l=0, Nq=0) == fa.FA_OK


def test_fp16_rejects_like_forward(lib):
    f = lib.fa_forward_fp16
    assert f(Q, K, V, O, L, 1, 3, 2, 64, 64, 128, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, 1, 2, 1, 64, 64, 96, 0, 0.1, None) == fa.FA_ERR_UNSUPPORTED
    assert f(Q, K, V, Q, L, 1, 2, 1, 64, 64, 128, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    assert f(Q + 8, K, V, O, L, 1, 2, 1, 64, 64, 128, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    assert f(0, 0, 0, 0, 0, 1, 2, 1, 0, 64, 128, 0, 0.1, None) == fa.FA_OK


def test_empty_query_is_a_no_op(lib):
    # nothing to write: success without touching the device (null pointers allowed)
    assert _fwd(lib, q=0, k=0, v=0, o=0, l=0, Nq=0) == fa.FA_OK
    assert _fwd(lib, q=0, k=0, v=0, o=0, l=0, B=0) == fa.FA_OK


def test_naive_rejects(lib):
    f = lib.fa_naive_forward
    need = lib.fa_naive_workspace_bytes(1, 2, 64, 64)
    W = 0x60000000
    assert f(Q, K, V, O, L, 1, 3, 2, 64, 64, 128, 0, 0.1, W, need, None) == fa.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, 1, 2, 1, 64, 64, 128, 0, 0.1, W, need - 1, None) == fa.FA_ERR_NO_MEMORY
    assert f(Q, K, V, O, L, 1, 2, 1, 64, 64, 128, 0, 0.1, 0, need, None) == fa.FA_ERR_NO_MEMORY
    assert f(Q, K, V, O, L, 1, 2, 1, 64, 64, 128, 0, 0.1, W + 8, need, None) == fa.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, 1, 2, 1, 64, 64, 128, 0, 0.1, O - 16, need, None) == fa.FA_ERR_INVALID_ARG
    assert f(Q, K, V, O, L, 1, 2, 1, 64, 64, 80, 0, 0.1, W, need, None) == fa.FA_ERR_UNSUPPORTED


def test_no_gpu_fails_loudly(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    # a valid request on a machine without a GPU is a CUDA error, never a silent success
    assert _fwd(lib) == fa.FA_ERR_CUDA


def test_selftest_rejects_limits_out_of_range(lib):
    # argument checks come before any CUDA call
    assert lib.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_wait_timeout(20_000_000_000, None) == fa.FA_ERR_INVALID_ARG


def test_binding_checks_element_types():
    # the binding refuses mixed or unsupported dtypes before anything reaches libfa
    torch = pytest.importorskip("torch")
    import exact_tiled_attention_forward_gb300 as fa
    q16 = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    qb = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    q32 = torch.zeros(1, 1, 8, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        fa.fa_forward(q16, qb, qb)                      # FP16 q, BF16 k and v
    with pytest.raises(TypeError):
        fa.fa_forward(qb, qb, qb, out=torch.zeros(1, 1, 8, 64, dtype=torch.float16))
    with pytest.raises(TypeError):
        fa.fa_forward(q32, q32, q32)                    # FP32 is not an element type here
    with pytest.raises(TypeError):
        fa.fa_forward_fp16(qb, qb, qb)
    with pytest.raises(TypeError):
        fa.fa_naive_forward(q16, q16, q16)
    with pytest.raises(TypeError):
        fa.fa_forward(qb, qb, qb, lse=torch.zeros(1, 1, 8, dtype=torch.float16))


def test_host_batch_rejects(lib):
    f = lib.fa_forward_host
    P = ctypes.c_void_p
    one = (P * 1)(0x1000)
    two = (P * 2)(0x1000, 0)                 # request 1 has a NULL pointer
    args = (1, 2, 1, 64, 64, 128, 0, 0.1, 0, None)
    assert f(0, None, None, None, None, None, *args) == fa.FA_OK          # nothing to do
    assert f(-1, one, one, one, one, None, *args) == fa.FA_ERR_INVALID_ARG
    assert f(1, None, one, one, one, None, *args) == fa.FA_ERR_INVALID_ARG
    assert f(2, two, two, two, two, None, *args) == fa.FA_ERR_INVALID_ARG
    assert f(1, one, one, one, one, None, 1, 3, 2, 64, 64, 128, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert f(1, one, one, one, one, None, 1, 2, 1, 64, 64, 96, 0, 0.1, 0, None) == fa.FA_ERR_UNSUPPORTED
    assert f(1, one, one, one, one, None, 1, 2, 1, 64, 64, 128, 0, float("nan"), 0, None) == fa.FA_ERR_INVALID_ARG
    assert f(1, one, one, one, one, None, 1, 2, 1, 64, 64, 128, 0, 0.1, 7, None) == fa.FA_ERR_INVALID_ARG
    # an empty query set is a no-op whatever the pointers
    assert f(1, (P * 1)(0), (P * 1)(0), (P * 1)(0), (P * 1)(0), None, 1, 2, 1, 0, 64, 128, 0, 0.1, 0,
             None) == fa.FA_OK


def test_host_batch_binding_checks():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16)
    o = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_forward_host([q], [k], [k, k], [o])                     # lists of unequal length
    with pytest.raises(ValueError):
        fa.fa_forward_host([q, q[:, :1].contiguous()], [k, k], [k, k], [o, o])   # shapes differ
    with pytest.raises(TypeError):
        fa.fa_forward_host([q], [k], [k], [o.half()])
    with pytest.raises(ValueError):
        fa.fa_forward_host([q.transpose(2, 3)], [k], [k], [o])       # not contiguous
    fa.fa_forward_host([], [], [], [])                                # nothing to do


def test_host_packed_rejects(lib):
    f = lib.fa_forward_host_packed
    P = ctypes.c_void_p
    one = (P * 1)(0x1000)
    assert f(0, None, None, 1, 2, 1, 64, 64, 128, 0, 0.1, 0, None) == fa.FA_OK
    assert f(-1, one, one, 1, 2, 1, 64, 64, 128, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert f(1, None, one, 1, 2, 1, 64, 64, 128, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert f(1, one, None, 1, 2, 1, 64, 64, 128, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert f(1, (P * 1)(0), one, 1, 2, 1, 64, 64, 128, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert f(1, one, one, 1, 2, 1, 64, 64, 80, 0, 0.1, 0, None) == fa.FA_ERR_UNSUPPORTED
    assert f(1, one, one, 1, 2, 1, 64, 64, 128, 0, 0.1, 2, None) == fa.FA_ERR_INVALID_ARG
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):       # a buffer too small for the shape
        fa.fa_forward_host_packed([torch.zeros(10, dtype=torch.uint8)], [torch.zeros(10, dtype=torch.uint8)],
                                  (1, 1, 1, 8, 8, 64))


def test_backward_rejects(lib):
    f = lib.fa_backward
    # q, k, v, o, lse, do, dq, dk, dv
    ok_ptrs = [0x10000000 * (i + 1) for i in range(9)]         # disjoint, 16-byte aligned
    args = (1, 2, 1, 64, 64, 128, 0, 0.1, 0, None)
    def call(**kw):
        p = list(ok_ptrs)
        for i, name in enumerate(["q", "k", "v", "o", "lse", "do", "dq", "dk", "dv"]):
            if name in kw:
                p[i] = kw[name]
        a = list(args)
        for i, name in enumerate(["B", "Hq", "Hkv", "Nq", "Nk", "d", "causal", "scale", "dtype"]):
            if name in kw:
                a[i] = kw[name]
        return f(*p, *a)
    assert call(Hq=3, Hkv=2) == fa.FA_ERR_INVALID_ARG
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert call(dtype=3) == fa.FA_ERR_INVALID_ARG
    assert call(lse=0) == fa.FA_ERR_INVALID_ARG                   # lse is required
    assert call(do=0x60000008) == fa.FA_ERR_INVALID_ARG            # misaligned
    assert call(dq=0x10000000 + 64) == fa.FA_ERR_INVALID_ARG       # dq overlaps q
    assert call(dk=0x70000000) == fa.FA_ERR_INVALID_ARG            # dk overlaps dq
    assert call(dv=0x30000000) == fa.FA_ERR_INVALID_ARG            # dv aliases v


def test_decode_paged_rejects(lib):
    f = lib.fa_decode_paged
    # q, k_cache, v_cache, block_table, seqlens, o, lse
    ok_ptrs = [0x10000000 * (i + 1) for i in range(7)]           # disjoint, 16-byte aligned
    names_p = ["q", "kc", "vc", "table", "lens", "o", "lse"]
    names_a = ["B", "Hq", "Hkv", "Nq", "pages", "max_pages", "d", "causal", "scale", "dtype"]
    args = (2, 8, 2, 1, 16, 4, 128, 0, 0.1, 0, None)

    def call(**kw):
        p = [kw.get(n, ok_ptrs[i]) for i, n in enumerate(names_p)]
        a = [kw.get(n, args[i]) for i, n in enumerate(names_a)] + [None]
        return f(*p, *a)
    assert call(Hq=3, Hkv=2) == fa.FA_ERR_INVALID_ARG
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(Nq=5) == fa.FA_ERR_UNSUPPORTED          # 4 heads x 5 rows per KV head > 16
    assert call(scale=float("inf")) == fa.FA_ERR_INVALID_ARG
    assert call(dtype=2) == fa.FA_ERR_INVALID_ARG
    assert call(pages=0) == fa.FA_ERR_INVALID_ARG
    assert call(max_pages=0) == fa.FA_ERR_INVALID_ARG
    assert call(table=0) == fa.FA_ERR_INVALID_ARG
    assert call(lens=0x50000002) == fa.FA_ERR_INVALID_ARG      # misaligned int32
    assert call(kc=0x20000008) == fa.FA_ERR_INVALID_ARG        # misaligned cache
    assert call(o=0x10000000 + 256) == fa.FA_ERR_INVALID_ARG   # o overlaps q
    assert call(lse=0x40000000) == fa.FA_ERR_INVALID_ARG       # lse overlaps the block table
    assert call(pages=1 << 29, Hkv=8, Hq=8) == fa.FA_ERR_INVALID_ARG   # page x head index past 31 bits
    assert call(B=0) == fa.FA_OK                                # nothing to do



def test_backward_binding_checks_layout(lib):
    torch = pytest.importorskip("torch")
    # the binding refuses tensors whose shape, layout or device would let libfa
    # read past a buffer (all raised before any call into libfa)
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 8)
    with pytest.raises(ValueError, match="do has shape"):
        fa.fa_backward(q, k, k, q, lse, torch.zeros(1, 2, 7, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="lse has shape"):
        fa.fa_backward(q, k, k, q, torch.zeros(1, 2, 9), q)
    with pytest.raises(ValueError, match="contiguous"):
        fa.fa_backward(q, k, k, q, lse, q.transpose(2, 3).contiguous().transpose(2, 3))
    with pytest.raises(ValueError, match="CUDA"):
        fa.fa_backward(q, k, k, q, lse, q)
    with pytest.raises(TypeError):
        fa.fa_backward(q, k, k, q, lse.double(), q)


def test_decode_paged_binding_checks_layout(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(2, 4, 1, 64, dtype=torch.bfloat16)
    kc = torch.zeros(3, 2, 128, 64, dtype=torch.bfloat16)
    table = torch.zeros(2, 2, dtype=torch.int32)
    lens = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(TypeError):
        fa.fa_decode_paged(q, kc, kc, table.long(), lens)
    with pytest.raises(ValueError, match="128"):
        fa.fa_decode_paged(q, kc[:, :, :64], kc[:, :, :64], table, lens)
    with pytest.raises(ValueError, match="block_table"):
        fa.fa_decode_paged(q, kc, kc, table[:1], lens)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fa_decode_paged(q, kc, kc, table, lens)
