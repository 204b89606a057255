"""Test infrastructure: the CPU oracle of the top-k / top-p logit filter.

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
package; the library never does.
"""
from .oracle import (  # noqa: F401
    F32, F16, BF16, apply, apply_row, apply_sorted, apply_sorted_row, decode,
    filter_sorted_row, neg_inf_bits, raw_bits, round_to_dtype_f32,
    sample, sample_row, stable_ascending_sort, top_p_threshold, topk_enabled, topk_survivors,
)
