"""GB300-native sparse decode: score -> exact top-k -> slot-table gather -> split-K attention.

The compute lives in libskv.so (hand-written sm_103a CUDA behind a C ABI,
declared in include/skv.h).  This package is its ctypes binding: the same
entry-point names, argument marshalling only.  Importing it fails if the
library has not been built -- there is no CPU fallback.
"""

from .binding import (  # noqa: F401
    SKV_AGG_HEAD,
    SKV_AGG_MAX,
    SKV_AGG_MEAN,
    SKV_DEV_BAD_INDEX,
    SKV_DEV_BAD_LENGTH,
    SKV_DEV_BAD_SLOT,
    SKV_DEV_TIMEOUT,
    SKV_DTYPE_BF16,
    SKV_DTYPE_F32,
    SKV_INDEX_CONTIG,
    SKV_INDEX_PAGED,
    IndexSrc,
    Pool,
    Paris,
    Prefetch,
    SlotCache,
    Problem,
    SkvError,
    lib,
    skv_block_decode_step,
    skv_block_select,
    skv_block_summaries,
    skv_block_workspace_size,
    skv_decode_step,
    skv_decode_step_cached,
    skv_paris_decode_step,
    skv_paris_encode,
    skv_paris_quantizer,
    skv_paris_select,
    skv_paris_workspace_offsets,
    skv_paris_workspace_size,
    skv_cache_update,
    skv_decode_step_prefetch,
    skv_gather,
    skv_check_wait_timeout,
    skv_launch_count,
    skv_score,
    skv_sparse_attn,
    skv_status_string,
    skv_topk,
    skv_workspace_size,
)
from .step import BlockStep, DecodeStep, ParisStep  # noqa: F401

lib()  # load now: a missing library is an import error, never a silent fallback
