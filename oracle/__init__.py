"""Float64 CPU oracle for exact online-softmax attention (test infrastructure).

Only tests, the smoke check and the benchmark's CPU-baseline legs may import
this package.  The CUDA library never imports, links or calls it.
"""
from .ref import (  # noqa: F401
    NEG_INF,
    all_orders_and_groupings,
    attention_bruteforce,
    attention_bwd_ref,
    attention_ref,
    finalize,
    lse_merge_ref,
    merge,
    merge_all,
    online_attention_single,
    online_attention_single_normalised,
    online_ml_trace,
    set_partitions,
    softmax_row_fsum,
    softmax_rows_ref,
    softmax_topk_ref,
    summary_of,
    tiled_softmax_online,
    visible_keys,
)
