"""GPU parity of the thread-block-cluster K/V multicast variant
(fa_forward_cluster_multicast, libfa_single_gpu.so, a one-GPU process only):
clusters of two CTAs of one head fetch each K/V tile once and multicast it into
both CTAs' shared memory. Same oracle and tolerances as the plain kernel;
includes pairs that straddle two heads (odd number of query blocks per head),
an idle CTA completing the last cluster, causal pairs with unequal key ranges,
GQA and ragged lengths. Results must also equal the plain kernel's bit for bit
(same arithmetic, only the loads differ)."""
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


def _run(fa, a, multicast):
    import torch
    fn = fa.fa_forward_cluster_multicast if multicast else fa.fa_forward
    o, lse = fn(to_dev(a.q), to_dev(a.k), to_dev(a.v), causal=a.causal, scale=a.scale)
    torch.cuda.synchronize()
    status = fa.lib_single_gpu().fa_device_status(1) if multicast else fa.fa_device_status()
    assert status == fa.FA_OK
    return bf16_dev_to_f64(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", [
    # (B, H_q, H_kv, N_q, N_k, d, causal); >= 152 query blocks so the plan has no split tail
    (1, 152, 152, 256, 640, 128, False),   # one block per head: every cluster straddles two heads
    (1, 76, 76, 512, 520, 128, False),     # two blocks per head: every cluster shares; ragged keys
    (2, 38, 38, 1024, 384, 64, False),     # d = 64, four blocks per head
    (1, 51, 51, 768, 768, 128, True),      # three blocks per head (odd): mixed; idle CTA at the end
    (2, 40, 10, 1000, 1000, 64, True),     # GQA, ragged, causal pairs with unequal ranges
    (1, 38, 38, 2048, 2048, 128, True),    # longer causal
])
def test_multicast_matches_oracle_and_plain(fa, shape):
    a = I.make_inputs(*shape[:6], causal=shape[6], seed=8, k_row_frac=0.01)
    o_mc, l_mc = _run(fa, a, True)
    o_pl, l_pl = _run(fa, a, False)
    assert np.array_equal(o_mc, o_pl) and np.array_equal(l_mc, l_pl)
    compare(o_mc, l_mc, *run_oracle(a))
