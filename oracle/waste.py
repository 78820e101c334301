"""Internal-fragmentation arithmetic of paged and contiguous KV caches.

Test infrastructure only.  Restates "Paged KV-Cache Memory Management"
(mini-infer), sections "The Problem" (the contiguous-reservation example) and
"Memory Waste Analysis" (the last-block bound).  The bound's formula is garbled
in the page's text; the reading used here is: a sequence of N tokens occupies
ceil(N/B) blocks, the unused slots all sit in its last block, and

    waste(N) = (ceil(N/B) * B - N) / N  <=  (B - 1) / N,

with equality exactly when N = 1 (mod B).
"""
from __future__ import annotations


def blocks_needed(n_tokens: int, block_size: int) -> int:
    return -(-n_tokens // block_size)


def paged_waste_fraction(n_tokens: int, block_size: int) -> float:
    """Reserved-but-unused slots over used slots for one sequence."""
    if n_tokens <= 0:
        raise ValueError("n_tokens must be positive")
    reserved = blocks_needed(n_tokens, block_size) * block_size
    return (reserved - n_tokens) / n_tokens


def paged_waste_bound(n_tokens: int, block_size: int) -> float:
    return (block_size - 1) / n_tokens


def contiguous_waste_fraction(reserved: int, used: int) -> float:
    """Fraction of a contiguous reservation left unused."""
    return (reserved - used) / reserved


def block_bytes(num_layers: int, num_kv_heads: int, block_size: int, head_dim: int,
                elem_bytes: int) -> int:
    """Bytes of one physical block: K and V rows of every layer and KV head."""
    return 2 * num_layers * num_kv_heads * block_size * head_dim * elem_bytes
