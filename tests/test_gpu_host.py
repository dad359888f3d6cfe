"""GPU: fa_forward_host and fa_forward_host_packed, requests whose tensors live
in host memory. Every request's O and LSE must equal fa_forward's on the same
inputs bit for bit (same kernels, same plan), and one request is checked against
the oracle."""
import numpy as np
import pytest

from exact_tiled_attention_forward_gb300 import inputs as I

from helpers import compare, run_oracle

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


def _host(torch, x, pin):
    t = torch.from_numpy(np.ascontiguousarray(x)) if x.dtype == np.float16 else \
        torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


def _requests(torch, shape, n, dtype, adjacent, pin):
    """n seeded requests as host tensors; with `adjacent` (the packed form), each
    request's Q|K|V are views of one buffer back to back, and so are O|LSE."""
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    reqs = [I.make_inputs(B, Hq, Hkv, Nq, Nk, d, causal=causal, seed=100 + i, dtype=dtype)
            for i in range(n)]
    el = torch.float16 if dtype == "f16" else torch.bfloat16
    qs, ks, vs, os_, ls, bufs = [], [], [], [], [], []
    for a in reqs:
        if adjacent:
            flat = np.concatenate([a.q.reshape(-1), a.k.reshape(-1), a.v.reshape(-1)])
            buf = _host(torch, flat, pin)
            nq, nk = a.q.size, a.k.size
            qs.append(buf[:nq].view(a.q.shape))
            ks.append(buf[nq:nq + nk].view(a.k.shape))
            vs.append(buf[nq + nk:].view(a.v.shape))
            ob = nq * 2
            out = torch.empty(ob + B * Hq * Nq * 4, dtype=torch.uint8)
            out = out.pin_memory() if pin else out
            os_.append(out[:ob].view(el).view(B, Hq, Nq, d))
            ls.append(out[ob:].view(torch.float32).view(B, Hq, Nq))
            bufs.append((buf, out))
        else:
            qs.append(_host(torch, a.q, pin))
            ks.append(_host(torch, a.k, pin))
            vs.append(_host(torch, a.v, pin))
            o = torch.empty(B, Hq, Nq, d, dtype=el)
            l = torch.empty(B, Hq, Nq, dtype=torch.float32)
            os_.append(o.pin_memory() if pin else o)
            ls.append(l.pin_memory() if pin else l)
    return reqs, qs, ks, vs, os_, ls, bufs


def _run(fa, reqs, qs, ks, vs, os_, ls, bufs, stream=None):
    a = reqs[0]
    if bufs:
        fa.fa_forward_host_packed([b[0] for b in bufs], [b[1] for b in bufs], a.shape_args,
                                  causal=a.causal, scale=a.scale, dtype=qs[0].dtype, stream=stream)
    else:
        fa.fa_forward_host(qs, ks, vs, os_, ls, causal=a.causal, scale=a.scale, stream=stream)


def _check_against_device_call(fa, torch, reqs, qs, ks, vs, os_, ls):
    for i, a in enumerate(reqs):
        o_ref, l_ref = fa.fa_forward(qs[i].cuda(), ks[i].cuda(), vs[i].cuda(), causal=a.causal,
                                     scale=a.scale)
        torch.cuda.synchronize()
        assert torch.equal(os_[i], o_ref.cpu()), f"request {i}: O differs from fa_forward"
        if ls is not None and ls[i] is not None:
            assert torch.equal(ls[i], l_ref.cpu()), f"request {i}: LSE differs from fa_forward"


CASES = [
    # (shape, n, dtype, adjacent, pinned)
    ((1, 4, 2, 700, 900, 128, True), 5, "bf16", False, True),    # three copies in, two out
    ((1, 4, 2, 700, 900, 128, True), 3, "bf16", True, True),     # packed: one copy each way
    ((1, 1, 1, 2048, 8192, 128, False), 3, "f16", True, True),   # split plan, FP16
    ((4, 8, 2, 1, 2048, 128, False), 4, "bf16", False, True),    # decode path
    ((4, 8, 2, 1, 2048, 128, False), 1, "bf16", False, True),    # one decode request
    ((4, 8, 2, 1, 2048, 128, False), 2, "f16", True, True),      # decode, packed, FP16
    ((1, 2, 2, 300, 300, 64, False), 1, "bf16", False, True),    # a single request: one slot
    ((1, 2, 1, 257, 513, 64, True), 3, "bf16", False, False),    # pageable host memory
]


@pytest.mark.parametrize("shape,n,dtype,adjacent,pin", CASES,
                         ids=lambda c: str(c) if not isinstance(c, tuple) else "x".join(map(str, c[:6])))
def test_host_requests_match_device_calls(fa, shape, n, dtype, adjacent, pin):
    import torch
    reqs, qs, ks, vs, os_, ls, bufs = _requests(torch, shape, n, dtype, adjacent, pin)
    for o in os_:
        o.fill_(-7.0)
    _run(fa, reqs, qs, ks, vs, os_, ls, bufs)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    _check_against_device_call(fa, torch, reqs, qs, ks, vs, os_, ls)
    o0 = os_[0].float().numpy().astype(np.float64)
    compare(o0, ls[0].numpy().astype(np.float64), *run_oracle(reqs[0]), elem=dtype)


def test_host_requests_without_lse(fa):
    import torch
    shape = (1, 2, 1, 500, 700, 128, False)
    reqs, qs, ks, vs, os_, ls, _ = _requests(torch, shape, 3, "bf16", False, True)
    fa.fa_forward_host(qs, ks, vs, os_, None, causal=False, scale=reqs[0].scale)
    torch.cuda.synchronize()
    _check_against_device_call(fa, torch, reqs, qs, ks, vs, os_, None)
    ls[1].fill_(5.0)
    fa.fa_forward_host(qs, ks, vs, os_, [ls[0], None, ls[2]], causal=False, scale=reqs[0].scale)
    torch.cuda.synchronize()
    assert torch.all(ls[1] == 5.0)                     # no LSE asked for: left alone
    _check_against_device_call(fa, torch, reqs, qs, ks, vs, os_, [ls[0], None, ls[2]])


def test_host_requests_follow_stream_order(fa):
    # work enqueued on the stream before the call runs first; work after it sees
    # the outputs in host memory once the stream is synchronised
    import torch
    shape = (1, 2, 2, 256, 1024, 128, True)
    reqs, qs, ks, vs, os_, ls, bufs = _requests(torch, shape, 4, "bf16", True, True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        busy = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
        busy.fill_(1)                                  # earlier work on the same stream
        _run(fa, reqs, qs, ks, vs, os_, ls, bufs, stream=s)
        done = torch.cuda.Event()
        done.record(s)
    done.synchronize()
    _check_against_device_call(fa, torch, reqs, qs, ks, vs, os_, ls)


def test_separate_tensors_in_one_buffer(fa):
    # separate-tensor form with Q, K, V (and O, LSE) that happen to be views of one
    # buffer: still copied one tensor at a time, results unchanged
    import torch
    shape = (1, 2, 1, 300, 500, 64, True)
    reqs, qs, ks, vs, os_, ls, _ = _requests(torch, shape, 3, "bf16", True, True)
    fa.fa_forward_host(qs, ks, vs, os_, ls, causal=True, scale=reqs[0].scale)
    torch.cuda.synchronize()
    _check_against_device_call(fa, torch, reqs, qs, ks, vs, os_, ls)
