"""Capacity and waste arithmetic of paged KV allocation.

Test infrastructure only (see the package docstring).

  * blocks per request = ceil(seq_len / block_size) (lux-666 notes
    "PagedAttention", "block size 是容量与 kernel 的共同参数").
  * Paged internal waste: only the last block of a sequence can be partly
    empty ("Phase 7 · Document 04 — PagedAttention", §2 "internal fragmentation
    drops ... at most one partially-filled block per sequence"; lux-666 notes,
    它为什么有效).
  * Naive waste: a request holds a contiguous slab sized for the maximum
    context (Document 04, §2 primer, the 100-token request in an 8k slab).
  * Capacity: concurrent sequences ~ pool blocks / blocks per sequence at the
    given context (Document 04, §4 "How experts reason", §11, §13 question 4).
"""

from __future__ import annotations

import numpy as np


def blocks_needed(seq_len: int, block_size: int) -> int:
    """Number of fixed-size blocks holding `seq_len` tokens."""
    if seq_len < 0 or block_size <= 0:
        raise ValueError("bad length or block size")
    q, r = divmod(int(seq_len), int(block_size))
    return q + (1 if r else 0)


def paged_internal_waste(seq_lens, block_size: int) -> float:
    """Fraction of reserved token slots left empty under paged allocation."""
    lens = [int(x) for x in seq_lens]
    reserved = sum(blocks_needed(L, block_size) * block_size for L in lens)
    if reserved == 0:
        return 0.0
    return (reserved - sum(lens)) / reserved


def naive_slab_waste(seq_lens, max_len: int) -> float:
    """Fraction of token slots left empty when each request holds a slab of
    `max_len` contiguous slots."""
    lens = [int(x) for x in seq_lens]
    reserved = len(lens) * int(max_len)
    if reserved == 0:
        return 0.0
    return (reserved - sum(lens)) / reserved


def concurrent_sequences(pool_blocks: int, context_len: int,
                         block_size: int) -> int:
    """Whole sequences of `context_len` tokens that fit in `pool_blocks`."""
    return int(pool_blocks) // blocks_needed(context_len, block_size)
