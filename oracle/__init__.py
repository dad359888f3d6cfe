"""FP64 CPU oracle for the exact attention forward — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it, and it
shares no code, header, table or constant with the CUDA library: the only
thing both sides consume is the seeded input buffer drawn by
``exact_tiled_attention_forward_gb300.inputs`` (which holds no attention
arithmetic).

Contents
--------
``attention``  the definition ``O = softmax(scale * Q K^T) V`` written out in
               FP64 with the score and probability matrices materialised
               (row block by row block), plus the per-row log-sum-exp; a
               tiled online-softmax restatement used as a self-check; a
               pure-Python brute force for tiny shapes; the split merge.
``traffic``    the pages' analytic HBM byte and FLOP counts.
``backward``   FP64 gradients dQ, dK, dV of the definition (chain rule, pinned by
               finite differences of the forward).
``paged``      decode over a paged K/V cache: each sequence's keys read out of
               its pages in order, then the definition.
``fp8``        FP8 E4M3 inputs: the exact value of each code, the definition
               on code * per-tensor factor, and the most that rounding P to
               E4M3 can move each output (the FP8 path's error term).

Every function names the page and section it follows. Each is pinned in
``tests/test_oracle_*.py`` against values the pages print, closed forms and
invariants (see the test files for the pin of each function).
"""
from .attention import (  # noqa: F401
    bf16_to_f64,
    to_f64,
    attention_reference,
    attention_rows,
    attention_tiled_online,
    online_softmax_blocks,
    brute_force_attention,
    merge_partials,
    visible_key_count,
)
from . import traffic  # noqa: F401
from .backward import attention_backward, backward_error_terms, forward_loss  # noqa: F401
from .paged import gather_sequence, paged_attention_reference  # noqa: F401
from .fp8 import attention_reference_fp8, e4m3_to_f64, p_rounding_bound_fp8, p_rounding_weight  # noqa: F401
