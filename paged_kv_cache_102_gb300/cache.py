"""PagedKVCache: one layer's paged K/V pools plus the host block manager.

A thin driver around the C ABI for callers that do not want to handle slot
mappings and copy pairs themselves.  Per decode step:

    slots, pairs = block_manager.append_slots(seq_ids)   # host (C++)
    paged_block_copy(pairs)                              # copy-on-write first
    paged_kv_append(k, v, slots)                         # then write the token
    paged_attention_decode(q, tables, lens)              # attend

Copies run before the append on the same stream: the diverging writer's new
block must hold the old tokens before its own token lands in it (iThome "how
to store the KV cache", section "Copy-on-Write").
"""
from __future__ import annotations

import numpy as np
import torch

from . import (PARTITION_AUTO, BlockManager, paged_attention_decode, paged_block_copy, paged_kv_append)


class PagedKVCache:
    def __init__(self, num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int,
                 dtype=torch.bfloat16, device="cuda", free_list=None, k_cache=None, v_cache=None,
                 k_scale=None, v_scale=None):
        self.num_blocks, self.num_kv_heads = num_blocks, num_kv_heads
        self.block_size, self.head_dim = block_size, head_dim
        self.device = torch.device(device)
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        self.k_cache = k_cache if k_cache is not None else torch.zeros(shape, dtype=dtype, device=self.device)
        self.v_cache = v_cache if v_cache is not None else torch.zeros(shape, dtype=dtype, device=self.device)
        self.k_scale, self.v_scale = k_scale, v_scale
        self.blocks = BlockManager(num_blocks, block_size, free_list=free_list)

    # -- host-side bookkeeping -------------------------------------------------
    def add_sequence(self, seq_id: int, num_tokens: int) -> None:
        """Allocate blocks for a request whose first num_tokens are already in the pool."""
        self.blocks.add_sequence(seq_id, num_tokens)

    def fork(self, parent_id: int, child_id: int) -> None:
        self.blocks.fork(parent_id, child_id)

    def free(self, seq_id: int) -> None:
        self.blocks.free_sequence(seq_id)

    def tables(self, seq_ids, max_blocks_per_seq=None):
        t, lens = self.blocks.tables(seq_ids, max_blocks_per_seq)
        return (torch.from_numpy(t).to(self.device, non_blocking=False),
                torch.from_numpy(lens).to(self.device, non_blocking=False))

    # -- device steps ------------------------------------------------------------
    def append(self, seq_ids, k: torch.Tensor, v: torch.Tensor, stream=None):
        """Write one new token per sequence (k, v: [n, Hkv, D]); returns (slots, cow pairs) on the host."""
        slots, pairs = self.blocks.append_slots(seq_ids)
        if len(pairs):
            paged_block_copy(self.k_cache, self.v_cache, torch.from_numpy(pairs).to(self.device), stream=stream)
        paged_kv_append(k, v, torch.from_numpy(slots).to(self.device), self.k_cache, self.v_cache,
                        self.k_scale, self.v_scale, stream=stream)
        return slots, pairs

    def decode(self, seq_ids, q: torch.Tensor, scale: float, out=None, partition_size=PARTITION_AUTO,
               max_blocks_per_seq=None, stream=None):
        tables, lens = self.tables(seq_ids, max_blocks_per_seq)
        return paged_attention_decode(q, self.k_cache, self.v_cache, tables, lens, scale, out=out,
                                      k_scale=self.k_scale, v_scale=self.v_scale,
                                      partition_size=partition_size, stream=stream)

    def unused_slots(self, seq_ids) -> int:
        """Slots allocated to these sequences but not yet written (tail waste)."""
        return int(sum(self.blocks.num_seq_blocks(s) * self.block_size - self.blocks.context_len(s)
                       for s in np.asarray(seq_ids)))
