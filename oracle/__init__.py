"""Float64 CPU oracle for speculative-draft decode attention.

Test infrastructure only: the tests, the smoke check and the benchmark's CPU
baseline use it; the product path never does.
"""
from .draft_attn_oracle import (  # noqa: F401
    MODES, SEG_FAR, SEG_LOCAL, Params, append_rotated_keys, attend, attend_group,
    fold_far_position, page_slot, rope, rope_angles, rope_inv_freq, round_to_bf16,
    select_keys, selection_list, sharp_gamma, tree_filter, window_start,
)
