"""Blocked (paged) KV cache and the append step (oracle).

Source: FastGen guide, "Paged KV Memory Management with Zero Overhead" - the KV
cache lives in non-contiguous fixed-size physical blocks addressed through
per-sequence block tables; paper summary page, Key points - a blocked KV cache
as in PagedAttention.

Layout (the library's too, stated independently): K and V caches are separate
arrays ``[num_blocks][H_kv][B][D]``.  Token position ``p`` of a sequence lives
in block ``table[p // B]`` at slot ``p % B``.

Storage values are kept as the raw storage type: ``float32`` for fp32 caches and
``uint16`` bit patterns for bf16 caches, so that appending is a bit copy and a
comparison is bit-exact.  Blocks are created lazily, zero-filled (a cache starts
at zero; slots nobody wrote stay zero).
"""
from __future__ import annotations

from typing import Dict, Iterable, Optional, Set

import numpy as np

from .composer import PassMeta


class BlockedCache:
    """A K or V cache stored block by block (only touched blocks exist)."""

    def __init__(self, num_heads_kv: int, block_size: int, head_dim: int, storage: np.dtype):
        self.num_heads_kv = int(num_heads_kv)
        self.block_size = int(block_size)
        self.head_dim = int(head_dim)
        self.storage = np.dtype(storage)
        self.blocks: Dict[int, np.ndarray] = {}

    def block(self, b: int) -> np.ndarray:
        blk = self.blocks.get(b)
        if blk is None:
            blk = np.zeros((self.num_heads_kv, self.block_size, self.head_dim), self.storage)
            self.blocks[b] = blk
        return blk

    def dense(self, num_blocks: int) -> np.ndarray:
        """The whole cache as ``[num_blocks][H_kv][B][D]`` (zeros where unwritten)."""
        out = np.zeros((num_blocks, self.num_heads_kv, self.block_size, self.head_dim), self.storage)
        for b, blk in self.blocks.items():
            out[b] = blk
        return out

    def gather(self, block_table: Iterable[int], length: int, head: int) -> np.ndarray:
        """Rows 0..length-1 of one KV head of one sequence, through its table."""
        table = list(block_table)
        rows = np.empty((length, self.head_dim), self.storage)
        B = self.block_size
        for p in range(length):
            rows[p] = self.block(table[p // B])[head, p % B]
        return rows


def kv_append(meta: PassMeta, k_new: np.ndarray, v_new: np.ndarray,
              k_cache: BlockedCache, v_cache: BlockedCache,
              only_seqs: Optional[Set[int]] = None) -> None:
    """Copy each pass token's K/V rows into its cache slot.

    For sequence s and its j-th new token (pass row ``q_start[s] + j``, position
    ``p = seen[s] + j``): ``cache[table_s[p // B]][h][p % B][:] = new[row][h][:]``
    for every KV head h.  ``k_new``/``v_new`` are ``[T][H_kv][D]`` in the cache's
    storage type.  ``only_seqs`` restricts the copy to some sequence ids (used
    for sampled checks of very large passes).
    """
    B = k_cache.block_size
    for s in range(meta.num_seqs):
        if only_seqs is not None and meta.seq_ids[s] not in only_seqs:
            continue
        table = meta.blocks_of(s)
        for j in range(meta.n_new[s]):
            row = meta.q_start[s] + j
            p = meta.seen[s] + j
            b, off = table[p // B], p % B
            k_cache.block(b)[:, off, :] = k_new[row]
            v_cache.block(b)[:, off, :] = v_new[row]
