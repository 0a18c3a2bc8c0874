"""KV-only byte accounting (oracle).

FADE-zh §使用注意事项 (3): ``compressed_storage_bytes()`` counts KV storage only (nvidia-smi
also counts weights). FADE-zh §配置预设 gives compression by preset (safe about 3-4x,
balanced about 5x, aggressive about 7-8x); §量化与Bit-Packing: INT2 V gives about 30% extra
compression; §性能基准 gives two measured KV sizes (Qwen2.5-3B 12.2 -> 4.0 MiB, Llama-3.2-1B
29.9 -> 6.3 MiB with about 29% evicted).

Layout being counted (the spec's): FP16 tokens store K and V at 2 bytes per channel; a middle
token stores d*k_bits/8 + d*v_bits/8 code bytes plus one fp16 scale per 32 channels for K and
for V. With product-quantised V (FADE-zh §产品量化) a middle token's V is d/4 code bytes and
no scale (the per-layer codebook, 256*d fp16 values, is a fixed cost counted apart). The FP16
baseline stores every token ever seen at 4*d bytes.
"""

from __future__ import annotations


def fp16_token_bytes(head_dim: int) -> int:
    return 4 * head_dim


def middle_token_bytes(head_dim: int, k_bits: int, v_bits: int, group: int = 32,
                       v_codec: str = "int") -> int:
    scales = 2 * (head_dim // group)
    if v_codec == "pq":
        return head_dim * k_bits // 8 + scales + head_dim // 4
    return head_dim * k_bits // 8 + scales + head_dim * v_bits // 8 + scales


def pq_codebook_bytes(head_dim: int) -> int:
    """One layer's PQ codebook: 256 centroids of every 4-channel sub-space, fp16."""
    return 256 * head_dim * 2


def unit_bytes(head_dim, n_fp16, n_mid, k_bits, v_bits) -> int:
    """Bytes held by one (layer, row, KV head)."""
    return n_fp16 * fp16_token_bytes(head_dim) + n_mid * middle_token_bytes(head_dim, k_bits, v_bits)


def compressed_bytes(layers, kv_heads, head_dim, n_sink, n_recent, n_mid, k_bits, v_bits,
                     rows=1) -> int:
    """Bytes of a whole cache whose rows all hold the same tier counts."""
    return layers * rows * kv_heads * unit_bytes(head_dim, n_sink + n_recent, n_mid, k_bits, v_bits)


def fp16_bytes(layers, kv_heads, head_dim, tokens, rows=1) -> int:
    return layers * rows * kv_heads * tokens * fp16_token_bytes(head_dim)
