"""fp64 CPU oracle for the sparse-decode step (test infrastructure, never the product path).

Only the test suite, the package smoke check and the benchmark's CPU-baseline leg
import this package.  It shares no code with the CUDA library.
"""

from .skv_oracle import *  # noqa: F401,F403
from .skv_oracle import (  # noqa: F401
    HeadTablePool,
    PagedPool,
    Problem,
    as_f64,
    attended_positions,
    block_attended_positions,
    block_regions,
    block_scores,
    block_summary,
    box_bound,
    cache_owner_from_table,
    cache_update,
    cache_update_heads,
    decode_unit_blocks,
    attention,
    attention_partial,
    bf16_bits_to_f64,
    decode_step_hbm_bytes,
    decode_head,
    decode_unit,
    echo_metadata_bytes,
    exact_topk,
    group_scores,
    fetch_time_s,
    group_query,
    lse_merge,
    prefetch_step,
    regions,
    scores,
    step_read_bytes,
)
