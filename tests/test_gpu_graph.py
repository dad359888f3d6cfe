"""libfa calls captured into CUDA graphs: a forward (whole blocks; key ranges
split and merged inside clusters; split and merged by the merge kernel with a
stream-ordered workspace; decode) and a backward are captured once on the
capture stream and replayed with new inputs copied into the captured buffers.
Every replay must reproduce a direct call on the same inputs bit for bit, and
one is checked against the FP64 oracle. One-time set-up (kernel attributes,
cluster-occupancy queries, the workspace pool, the status word) happens on a
first call made before the capture, as graph capture requires."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import compare, run_oracle, to_dev

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


FWD = [
    # (B, H_q, H_kv, N_q, N_k, d, causal), FA_CLUSTER_MERGE
    ((1, 8, 8, 1024, 1024, 128, True), "1"),     # whole blocks
    ((1, 1, 1, 2048, 8192, 128, False), "1"),    # split key ranges, in-cluster merge
    ((1, 1, 1, 2000, 3000, 64, False), "0"),     # split, merge kernel, workspace from the pool
    ((4, 32, 8, 1, 6000, 64, False), "1"),       # decode
    ((1, 8, 2, 1, 40000, 128, False), "1"),      # decode, merge kernel
]


@pytest.mark.parametrize("shape,cm", FWD, ids=lambda x: "x".join(map(str, x[:6])) if isinstance(x, tuple) else f"cm{x}")
def test_forward_graph_replay(fa, shape, cm, monkeypatch):
    import torch
    monkeypatch.setenv("FA_CLUSTER_MERGE", cm)
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    runs = [I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=40 + i, k_row_frac=0.01) for i in range(3)]
    q, k, v = to_dev(runs[0].q), to_dev(runs[0].k), to_dev(runs[0].v)
    o = torch.empty(B, Hq, Nq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device="cuda")
    scale = runs[0].scale
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # the first call (one-time set-up) outside the capture
        fa.fa_forward(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.fa_forward(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
    torch.cuda.synchronize()
    for i, a in enumerate(runs):
        q.copy_(to_dev(a.q)); k.copy_(to_dev(a.k)); v.copy_(to_dev(a.v))
        o.fill_(7.0); lse.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_device_status() == fa.FA_OK
        og, lg = o.clone(), lse.clone()
        od, ld = fa.fa_forward(q, k, v, causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(og, od) and torch.equal(lg, ld)
        if i == 0:
            compare(og.float().cpu().numpy().astype(np.float64), lg.cpu().numpy().astype(np.float64), *run_oracle(a))


def test_backward_graph_replay(fa):
    import torch
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 300, 700, 128
    runs = [I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=True, seed=50 + i) for i in range(2)]
    q, k, v = to_dev(runs[0].q), to_dev(runs[0].k), to_dev(runs[0].v)
    do = to_dev(I.grad_output(runs[0], seed=50))
    o, lse = fa.fa_forward(q, k, v, causal=True, scale=runs[0].scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fa.fa_backward(q, k, v, o, lse, do, causal=True, scale=runs[0].scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.fa_forward(q, k, v, causal=True, scale=runs[0].scale, out=o, lse=lse)
        fa.fa_backward(q, k, v, o, lse, do, causal=True, scale=runs[0].scale, dq=dq, dk=dk, dv=dv)
    for i, a in enumerate(runs):
        q.copy_(to_dev(a.q)); k.copy_(to_dev(a.k)); v.copy_(to_dev(a.v))
        do.copy_(to_dev(I.grad_output(a, seed=50 + i)))
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_device_status() == fa.FA_OK
        got = [dq.clone(), dk.clone(), dv.clone()]
        o2, l2 = fa.fa_forward(q, k, v, causal=True, scale=a.scale)
        ref = fa.fa_backward(q, k, v, o2, l2, do, causal=True, scale=a.scale)
        torch.cuda.synchronize()
        for x, y in zip(got, ref):
            assert torch.equal(x, y)
        if i == 0:
            refs = oracle.attention_backward(a.q, a.k, a.v, I.grad_output(a, seed=50), causal=True, scale=a.scale)
            for x, r in zip(got, refs):
                x = x.float().cpu().numpy().astype(np.float64)
                assert np.linalg.norm(x - r) / np.linalg.norm(r) <= 1e-2
