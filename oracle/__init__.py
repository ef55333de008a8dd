"""Test infrastructure: the float64 CPU oracle for attention over a paged KV cache.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
legs may import this package.  It shares no code with the CUDA library.
Every function cites the passage of the pages it follows; see
``oracle/paged_attention.py``.
"""
from .paged_attention import (  # noqa: F401
    BF16_ATOL, BF16_REL_OF_MAX, FP32_ATOL, attend, decode, decode_partials, gather_kv,
    kv_write, merge_partials, narrow, prefill, qk_norm_rope, reference_step, rms_norm,
    rope, rope_inv_freq, round_to_bf16, round_to_dtype, slot_mapping, widen,
    within_tolerance)
