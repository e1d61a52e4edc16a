"""Storage arithmetic of the quantized KV cache (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description,
storage paragraph: K+V bytes per token per KV head at head_dim 256, and the whole-cache totals for
a 262,144-token, 16-layer, 4-KV-head cache.

A quantized row costs its packed codes plus one fp16 scale; an fp16 row costs 2 bytes per element.
"""
from __future__ import annotations

from .symmetric import packed_dim


def row_bytes(head_dim: int, bits: int) -> int:
    """Bytes of one stored (token, KV head) row: 16 -> plain fp16; 8/6/4 -> packed + fp16 scale."""
    if bits == 16:
        return 2 * head_dim
    return packed_dim(head_dim, bits) + 2


def kv_bytes_per_token_head(head_dim: int, bits: int) -> int:
    """K plus V bytes per token per KV head."""
    return 2 * row_bytes(head_dim, bits)


def cache_bytes(tokens: int, layers: int, kv_heads: int, head_dim: int, bits: int) -> int:
    return tokens * layers * kv_heads * kv_bytes_per_token_head(head_dim, bits)
