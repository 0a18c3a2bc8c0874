"""FADE tiered KV cache: decode attention on one GB300 (sm_103a) through the libfade C ABI."""

from .fade import (  # noqa: F401
    Config,
    FadeError,
    TieredLayer,
    fade_cache_append,
    fade_cache_demote,
    fade_cache_prefill,
    fade_cache_reset,
    fade_compressed_bytes,
    fade_decode_attention,
    fade_dequantize,
    fade_evict_rerope,
    fade_h2o_accumulate,
    fade_last_error,
    fade_layout,
    fade_next_position,
    fade_quantize_pack,
    fade_rope_apply,
    fade_rope_table_init,
    lib,
    preset,
)
