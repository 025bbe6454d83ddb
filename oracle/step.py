"""One decode step, end to end, on the CPU.

Test infrastructure only (see the package docstring).

Order of a step (the plain reading of "one decode step plus one append per
sequence"): the block manager reserves each sequence's next slot (growing the
table or copying a shared block first), the copy-on-write copies run, the new
K/V rows are written, then every sequence attends over its cached tokens
including the one just appended.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

from .allocator import BlockAllocator
from .attention import decode_attention
from .cache_ops import append_kv, copy_blocks


@dataclass
class DecodeStepResult:
    allocator: BlockAllocator
    slot_mapping: np.ndarray      # int32 [S]
    cow_pairs: np.ndarray         # int32 [n][2] (src, dst)
    block_table: np.ndarray       # int32 [S][MB], -1 past each sequence's blocks
    seq_lens: np.ndarray          # int32 [S], tokens attended
    k_pool: np.ndarray            # fp16 pools after copy + append
    v_pool: np.ndarray
    out: Optional[np.ndarray]     # fp64 [S][Hq][D] (None if not computed)


def place_batch(batch) -> BlockAllocator:
    """Replay the batch's churn, then register sequence i with its prefill."""
    a = BlockAllocator(batch.num_blocks, batch.block_size, batch.free_order)
    for op in batch.churn:
        if op.kind == "alloc":
            a.add_seq(op.owner, op.nblocks * batch.block_size)
        else:
            a.free_seq(op.owner)
    for i in range(batch.num_seqs):
        a.add_seq(i, int(batch.prefill_lens[i]))
    return a


def decode_step(batch, max_blocks: Optional[int] = None,
                compute_attention: bool = True, seqs=None,
                heads=None) -> DecodeStepResult:
    a = place_batch(batch)
    S = batch.num_seqs
    slots = np.empty(S, dtype=np.int32)
    pairs = []
    for i in range(S):
        slot, src, dst = a.append_slot(i)
        slots[i] = slot
        if src >= 0:
            pairs.append((src, dst))
    pairs_arr = np.array(pairs, dtype=np.int32).reshape(-1, 2)
    kp, vp = batch.k_pool, batch.v_pool
    if len(pairs):
        kp, vp = copy_blocks(kp, vp, pairs_arr)
    kp, vp = append_kv(kp, vp, batch.k_new, batch.v_new, slots)
    lens = np.array([a.seq_len(i) for i in range(S)], dtype=np.int32)
    mb = max_blocks if max_blocks is not None else \
        max(1, max(len(a.table(i)) for i in range(S)))
    table = np.array(a.dense_table(range(S), mb, fill=-1), dtype=np.int32)
    out = None
    if compute_attention:
        out = decode_attention(batch.q, kp, vp, table, lens, batch.scale,
                               seqs=seqs, heads=heads)
    return DecodeStepResult(a, slots, pairs_arr, table, lens, kp, vp, out)
