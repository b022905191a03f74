"""CPU fp64 oracle for Top-K block-sparse routed attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
the benchmark's CPU-baseline / reference leg may import this package.  The
CUDA library never calls it and shares no code with it.
"""

from .oracle import (  # noqa: F401
    BLOCK,
    HEAD_DIM,
    Sizes,
    block_lists,
    centroids,
    check_key_bias,
    decode_bf16,
    dense_score_bytes,
    derive_sizes,
    forward,
    forward_rows,
    kept_flops,
    kept_keys_per_row,
    local_video_blocks,
    plan,
    route_scores,
    row_key_set,
    select_topk,
    topk_count,
)
from .spark import (  # noqa: F401
    bf16_bits,
    block_ranges,
    forward_merged,
    reweight_bytes,
    round_to_bf16,
    skipped_blocks,
    spark_forward,
    spark_reweight,
    video_query_anchor,
)
from .reblock import reblock_bytes, spark_reblock  # noqa: F401
