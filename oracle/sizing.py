"""Pool-sizing arithmetic of the paged KV cache (test infrastructure only).

"11. Paged attention 与 online softmax" (dilfish.github.io), §11.1: a sequence
of T tokens needs ceil(T/B) blocks per layer and L*ceil(T/B) over L layers; a
pool of numBlocks blocks holds numBlocks * B * 2 * kvDim * elt bytes (K and V);
the last block of a sequence holds T - B*(ceil(T/B) - 1) tokens.

"从零开始写Qwen3（六）PagedAttention" (mlqm.cn), section "KVCache大小计算":
one token costs 2 (K and V) * layers * (kv heads * head_dim) * elt bytes.
"""
from __future__ import annotations


def blocks_per_layer(T: int, B: int) -> int:
    return -(-T // B)


def pool_blocks(T: int, B: int, L: int) -> int:
    return L * blocks_per_layer(T, B)


def pool_bytes(num_blocks: int, B: int, kv_dim: int, elt: int) -> int:
    return num_blocks * B * 2 * kv_dim * elt


def tokens_in_last_block(T: int, B: int) -> int:
    return T - B * (blocks_per_layer(T, B) - 1)


def kv_bytes_per_token(layers: int, kv_dim: int, elt: int) -> int:
    return 2 * layers * kv_dim * elt
