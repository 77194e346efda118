"""Float64 CPU oracle for range-masked attention -- test infrastructure only.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may import
anything from here; the product path never does.  See ``ffa_oracle`` for what it computes
and which passages it follows.
"""
from .ffa_oracle import (  # noqa: F401
    CAUSAL, FULL, TILE_EMPTY, TILE_FULL, TILE_PARTIAL, backward, dense_mask, forward, gather_pages,
    key_intervals, lse_merge, mask_block, normalize_slices, resolve_scale, row_intervals,
    tile_classes, visible_pairs,
)
