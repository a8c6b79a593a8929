"""Block and pool sizing (oracle, test infrastructure only).

Source: "PagedAttention Memory Management" (apxml course page), section
"Calculating Physical Block Sizes": one physical block holds the keys and the
values of T_block consecutive tokens for every layer and KV head, so its size
is the product 2 * L * N_kv * D_head * T_block * P_bytes (the 2 counts K and
V; P_bytes is 2 for FP16/BF16 and 1 for FP8).  The pool is the KV budget
divided into whole blocks.

Source for the per-sequence bookkeeping: the foundry page on paged block
allocation, "Concept" (blocks are allocated on demand, one per block_size
tokens, so the waste is at most block_size - 1 tokens) and the katajob Q&A,
"The paging idea" (a sequence gains one block every block_size tokens).
"""
from __future__ import annotations


def block_bytes(num_layers: int, num_kv_heads: int, head_dim: int, block_size: int,
                elem_bytes: int) -> int:
    """Bytes of one physical block: 2 * L * N_kv * D_head * T_block * P_bytes."""
    for v in (num_layers, num_kv_heads, head_dim, block_size, elem_bytes):
        if int(v) <= 0:
            raise ValueError("block size factors must be positive")
    return 2 * num_layers * num_kv_heads * head_dim * block_size * elem_bytes


def num_blocks_for_budget(budget_bytes: int, bytes_per_block: int) -> int:
    """Whole blocks that fit a KV budget (the pool is carved into blocks)."""
    if bytes_per_block <= 0:
        raise ValueError("block bytes must be positive")
    return int(budget_bytes) // int(bytes_per_block)


def blocks_for_tokens(num_tokens: int, block_size: int) -> int:
    """Blocks a sequence of num_tokens holds when blocks are taken on demand:
    the smallest count whose capacity covers the tokens."""
    n = 0
    while n * block_size < num_tokens:
        n += 1
    return n


def paged_waste_tokens(num_tokens: int, block_size: int) -> int:
    """Reserved-but-unwritten token slots of one sequence under paging."""
    return blocks_for_tokens(num_tokens, block_size) * block_size - num_tokens


def contiguous_waste_tokens(reserved_tokens: int, used_tokens: int) -> int:
    """Empty slots of the pre-paging design, one slab reserved per request."""
    return reserved_tokens - used_tokens


def shareable_prefix_tokens(prefix_tokens: int, block_size: int) -> int:
    """Tokens of a common prefix that whole-block sharing can reuse: sharing is
    block-granular, so only the filled blocks of the prefix are shared (the
    foundry page, "Failure modes", prefix hit rate)."""
    return (prefix_tokens // block_size) * block_size
