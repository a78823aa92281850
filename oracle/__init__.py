"""Plain float64 CPU oracle for context-parallel striped paged attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it.  It shares no code with the
CUDA library (no kernels, headers, helpers, tables or pre/post-processing); the
only thing both sides consume is the seeded input generator, which holds none
of the method's arithmetic.

Every function follows a passage of the source pages:

* mstar PR #1124 "Context / Sequence Parallel 1/5" (description; review thread
  on resident planning and on captured-bucket padding) -- the striped placement,
  per-partner partial with log-sum-exp, exact merge, own-token attention of
  non-decode steps, padding that merges to zero.
* vLLM "[Core] Add explicit layer parallel plans",
  ``vllm/v1/attention/backends/flash_attn.py``, ``FlashAttentionImpl.
  _forward_with_dcp`` -- context partial over the paged cache, own-token
  partial with ``cu_seqlens_k = cu_seqlens_q`` (causal), ``merge_attn_states``,
  the per-tensor ``k_descale`` / ``v_descale`` of an FP8 KV cache, and the
  interleave size ``cp_kv_cache_interleave_size`` (FlashAttentionMetadataBuilder).

Pinning status (what each function is checked against, in
``tests/test_oracle_pins.py``): every public function has at least one pin
that does not go through the function itself (brute force, closed forms, a
library routine, hand-derived golden fixtures, bijection/invariant checks).
No function here is "parity unpinned".
"""

from .reference import (  # noqa: F401
    E4M3_MAX,
    NEG_INF,
    attention,
    bf16_bits_to_f64,
    causal_own_attention,
    e4m3_dequantize,
    e4m3_encode,
    e4m3_quantize,
    e4m3_table,
    e4m3_value,
    expected_pool_image,
    expected_step,
    merge,
    mla_kv,
    placement,
    placement_inverse,
    raw_to_f64,
    stripe_partial,
    stripe_positions,
)
