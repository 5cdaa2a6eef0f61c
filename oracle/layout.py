"""Latent-cache footprint and the paged layout (oracle, test infrastructure only).

Footprint: a latent-attention layer caches one latent per token, of
kv_lora_rank + qk_rope_head_dim elements, plus the sparse-attention indexer key
when the model has one; linear-attention layers cache nothing.
Source: "hf: size GLM-5.3-Flash's KV cache from its latent layers only" (#64),
PR description (the two fixes and the sizing paragraph; DeepSeek V2/V3/V3.2 fall
to 576 per layer).

Paged layout (reading adopted for the paged cache): physical block p holds
``block_size`` consecutive token slots; token position t of sequence b lives in
block ``block_table[b][t // block_size]`` at slot ``t % block_size``. Within a
slot the bf16/fp32 kind stores [latent (r) | rope key (d_R)]; the rotated INT2
kind stores codes, scale/zero pairs and the rope key in three separate arrays
with the same block/slot indexing.
"""
from __future__ import annotations

import numpy as np


def footprint_elems(kv_lora_rank: int, qk_rope_head_dim: int, index_head_dim: int = 0) -> int:
    """Elements cached per token per latent-attention layer."""
    return kv_lora_rank + qk_rope_head_dim + index_head_dim


def kv_bytes_per_token(layer_types, kv_lora_rank: int, qk_rope_head_dim: int,
                       index_head_dim: int = 0, bytes_per_elem: int = 2) -> int:
    """Bytes of cache per token across a model's layers.

    ``layer_types`` lists each layer as "linear_attention" (no growing cache) or
    any other string (a latent-attention layer).
    """
    per_layer = footprint_elems(kv_lora_rank, qk_rope_head_dim, index_head_dim)
    n_latent = sum(1 for t in layer_types if t != "linear_attention")
    return n_latent * per_layer * bytes_per_elem


def write_paged(num_blocks: int, block_size: int, width: int, block_table: np.ndarray,
                rows_per_seq, start_pos, dtype=np.float32, fill=0) -> np.ndarray:
    """Place each sequence's rows at positions start_pos[b], start_pos[b]+1, ...

    Returns the pool as [num_blocks, block_size, width]. Slots no sequence writes
    keep ``fill``.
    """
    pool = np.full((num_blocks, block_size, width), fill, dtype=dtype)
    for b, rows in enumerate(rows_per_seq):
        for i in range(rows.shape[0]):
            t = int(start_pos[b]) + i
            blk = int(block_table[b, t // block_size])
            pool[blk, t % block_size, :] = rows[i]
    return pool


def read_paged(pool: np.ndarray, block_table_row: np.ndarray, L: int, block_size: int) -> np.ndarray:
    """Gather the first L token rows of one sequence from the pool, in position order."""
    out = np.empty((L,) + pool.shape[2:], dtype=pool.dtype)
    for t in range(L):
        out[t] = pool[int(block_table_row[t // block_size]), t % block_size]
    return out
