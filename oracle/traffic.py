"""The pages' analytic HBM-byte and FLOP models (test infrastructure only).

Each function restates one model the pages compute, in the pages' units:

* "FlashAttention HBM bytes, one head, 8K" (inferenceinterviews.com),
  section "A strong answer": compulsory bytes (Q, K, V read and O written
  once), naive unfused traffic (S written, read, P written, read), the
  FlashAttention-2 "paper model" in which every query block re-reads all of K
  and V, FLOPs ``4 N^2 d``, intensity, and times at a given bandwidth or
  throughput. Section "What interviewers probe next": causal halves the
  FLOPs; decode reads K and V once per KV head for ``4 N d`` FLOPs per query
  head.
* "Flash Attention Mechanics: How Tiled Attention Fits in SRAM"
  (interviewprepkit.dev): section "Why Standard Attention Is Memory-Bound"
  (memory footprint of standard vs flash attention), section "SRAM
  Constraints and Block Size Selection" (per-SM tile bytes and intensity per
  inner step) and section "HBM Traffic Reduction" (traffic with Q, K, V, O
  touched once; largest context in a memory budget).
* "Why is standard attention memory-bound, and how does FlashAttention fix
  it?" (interview.clozo.ai), Steps 2 and 3: standard traffic (four passes over
  the score matrix plus Q, K, V, O) and the tiled traffic of a K/V-outer
  loop that reads K and V once and re-reads Q and O on each of ``N / B_c``
  passes, with ``B_c = M / (4 d)`` for an SRAM of ``M`` numbers.

MiB/GiB are binary (2^20, 2^30); MB and TB/s are decimal, as on page 1,
"Common mistakes".
"""
from __future__ import annotations

MIB = 1 << 20
GIB = 1 << 30


# ---- page 1: one head, FA2 order -------------------------------------------------

def tensor_bytes(n: int, d: int, elem: int = 2) -> int:
    """One N x d tensor."""
    return n * d * elem


def compulsory_bytes(n_q: int, n_k: int, d: int, elem: int = 2, h_q: int = 1,
                     h_kv: int | None = None, batch: int = 1) -> int:
    """Floor for any kernel: read Q, K, V once (K, V once per KV head), write O once."""
    h_kv = h_q if h_kv is None else h_kv
    return batch * elem * d * (2 * h_q * n_q + 2 * h_kv * n_k)


def naive_score_bytes(n_q: int, n_k: int, elem: int = 2) -> int:
    """The materialised score matrix S of one head."""
    return n_q * n_k * elem


def naive_traffic_bytes(n_q: int, n_k: int, d: int, elem: int = 2, score_elem: int | None = None) -> int:
    """Unfused: write S, read S, write P, read P (4 passes) plus the compulsory bytes."""
    se = elem if score_elem is None else score_elem
    return 4 * naive_score_bytes(n_q, n_k, se) + compulsory_bytes(n_q, n_k, d, elem)


def paper_model_bytes(n: int, d: int, block_rows: int, elem: int = 2) -> int:
    """FA2 paper model: each of the ``N / B_r`` query blocks re-reads all of K and V;
    Q read once and O written once."""
    t_r = n // block_rows
    return t_r * 2 * tensor_bytes(n, d, elem) + 2 * tensor_bytes(n, d, elem)


def forward_flops(n_q: int, n_k: int, d: int, causal: bool = False, h_q: int = 1,
                  batch: int = 1) -> float:
    """``4 N_q N_k d`` per query head (QK^T and PV), halved when causal."""
    f = 4.0 * n_q * n_k * d * h_q * batch
    return f / 2 if causal else f


def intensity(flops: float, nbytes: float) -> float:
    return flops / nbytes


def seconds(amount: float, rate: float) -> float:
    """Time to move ``amount`` bytes (or do ``amount`` FLOPs) at ``rate`` per second."""
    return amount / rate


def decode_kv_bytes_per_kv_head(n_k: int, d: int, elem: int = 2) -> int:
    """Decode reads K and V of one KV head once."""
    return 2 * tensor_bytes(n_k, d, elem)


def decode_flops_per_query_head(n_k: int, d: int) -> float:
    """One query against ``n_k`` keys: ``4 n_k d`` FLOPs (scores and weighted sum)."""
    return 4.0 * n_k * d


# ---- page 2: footprint, SRAM, traffic tables (32 heads, d = 128) -----------------

def standard_footprint_bytes(n: int, heads: int, d: int, elem: int = 2) -> int:
    """Score matrix + Q, K, V + output."""
    return heads * n * n * elem + 3 * heads * n * d * elem + heads * n * d * elem


def flash_footprint_bytes(n: int, heads: int, d: int, elem: int = 2) -> int:
    """Q, K, V, O plus two statistics per row (sized with the tensors' element
    width, as the page's table is)."""
    return 4 * heads * n * d * elem + heads * n * 2 * elem


def sram_tile_bytes(block: int, d: int, elem: int = 2) -> int:
    """Q, K, V and O tiles of ``block`` rows plus FP32 m and l per row."""
    return 4 * block * d * elem + block * 2 * 4


def tile_intensity(block: int, d: int, elem: int = 2) -> float:
    """FLOPs of one inner step (``4 B^2 d``) over the K and V tile bytes."""
    return 4.0 * block * block * d / (2 * block * d * elem)


def best_block(sram_bytes: int, d: int, candidates=(16, 32, 64, 128, 256, 512)) -> int:
    """Largest candidate block whose tiles fit the SRAM budget."""
    fit = [b for b in candidates if sram_tile_bytes(b, d) <= sram_bytes]
    return max(fit) if fit else 0


def standard_traffic_bytes(n: int, heads: int, d: int, elem: int = 2) -> int:
    """Four passes over the score matrix plus Q, K, V read and O written."""
    return 4 * heads * n * n * elem + 4 * heads * n * d * elem


def flash_traffic_bytes(n: int, heads: int, d: int, elem: int = 2) -> int:
    """Q, K, V, O each touched once."""
    return 4 * heads * n * d * elem


def max_context(heads: int, d: int, budget_bytes: int, flash: bool,
                candidates=(2048, 4096, 8192, 16384, 32768, 65536, 131072, 262144)) -> int:
    """Largest candidate length whose attention activations fit the budget:
    the N x N scores for standard attention, Q, K, V, O for flash."""
    best = 0
    for n in candidates:
        need = 4 * heads * n * d * 2 if flash else heads * n * n * 2
        if need <= budget_bytes:
            best = n
    return best


# ---- page 3: K/V-outer (FA1-order) tiled model ------------------------------------

def p3_standard_bytes(n: int, d: int, elem: int = 2) -> int:
    """Four passes over one head's N x N matrix plus Q, K, V, O."""
    return 4 * n * n * elem + 4 * n * d * elem


def p3_block_cols(sram_numbers: int, d: int) -> int:
    """``B_c = M / (4 d)`` columns for an SRAM of ``M`` numbers."""
    return sram_numbers // (4 * d)


def p3_tiled_bytes(n: int, d: int, sram_numbers: int, elem: int = 2) -> int:
    """K and V read once; each of the ``N / B_c`` passes reads Q, reads O and writes O."""
    passes = n // p3_block_cols(sram_numbers, d)
    return 2 * tensor_bytes(n, d, elem) + passes * 3 * tensor_bytes(n, d, elem)
