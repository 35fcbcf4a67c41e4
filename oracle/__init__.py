"""CPU oracle (test infrastructure; never imported by the product path)."""
from .ragged_attention import (  # noqa: F401
    attend,
    attend_row,
    cls_scores,
    cls_weights,
    linear_packed,
    pack_indices,
    pack_rows,
    pipeline,
    topk_keep,
    unpack,
)
