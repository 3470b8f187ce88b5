"""Byte and page counting (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""
from __future__ import annotations


def kv_cache_bytes(layers: int, batch: int, heads: int, seq_len: int, head_dim: int,
                   bytes_per_elem: int) -> int:
    """layers x 2 (K and V) x batch x heads x seq_len x head_dim x bytes.

    [KV-practice page, section 2.1]: each layer caches K and V of shape
    [batch, heads, seq_len, dim].
    """
    return layers * 2 * batch * heads * seq_len * head_dim * bytes_per_elem


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """ceil(num_tokens / block_size) [HBM-layout page, section 三 allocate_blocks]."""
    return (num_tokens + block_size - 1) // block_size
