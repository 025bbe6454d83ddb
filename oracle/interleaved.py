"""The one-pool layout of the layout sketch: each physical block is one record
holding its K array and then its V array.

Test infrastructure only (see the package docstring).

"Phase 7 · Document 04 — PagedAttention", §2 Core Concept, sketches the pool
as an array of physical-block records, each record a K array of
[BLOCK][HEADS][HEAD_DIM] halves followed by a V array of the same shape. The
other modules of this package keep K and V in two pools of [num_blocks][BS]
[Hkv][D]; here both live in one array of records.

Readings where the sketch leaves a step open:
  * The record is laid out as a C compiler lays out a struct of two arrays of
    one element type: K at byte offset 0, V right after it at BS*Hkv*D
    elements, no padding (both members have the element's alignment, and the
    record's size is already a multiple of it). Record b starts at
    b * 2*BS*Hkv*D elements.
  * HEADS is the number of KV heads, as in the two-pool layout.
  * The same record with one-byte elements holds an E4M3 cache (the fp8
    reading of `fp8.py`).
  * Every operation means what it means on the two-pool layout with K :=
    the records' K members and V := their V members: a slot is (record
    slot // BS, row slot % BS) of both members; a block copy copies the whole
    record.

The record type is a numpy structured dtype, which uses C's struct layout
rule; the tests pin it against byte offsets computed from that rule.
"""

from __future__ import annotations

import numpy as np

from .attention import decode_attention
from .fp8 import decode_attention_fp8


def kv_block_dtype(block_size: int, num_kv_heads: int, head_dim: int, elem=np.float16) -> np.dtype:
    """The record of one physical block: K[BS][Hkv][D] then V[BS][Hkv][D]."""
    shape = (int(block_size), int(num_kv_heads), int(head_dim))
    return np.dtype([("K", elem, shape), ("V", elem, shape)])


def make_kv_pool(k_pool: np.ndarray, v_pool: np.ndarray) -> np.ndarray:
    """The one-pool array of records holding the blocks of two separate pools
    ([NB][BS][Hkv][D] each): record b has K = k_pool[b] and V = v_pool[b]."""
    nb, bs, h, d = k_pool.shape
    kv = np.zeros(nb, dtype=kv_block_dtype(bs, h, d, k_pool.dtype))
    kv["K"] = k_pool
    kv["V"] = v_pool
    return kv


def split_kv_pool(kv_pool: np.ndarray) -> tuple:
    """(K, V) as [NB][BS][Hkv][D] arrays (views into the records)."""
    return kv_pool["K"], kv_pool["V"]


def append_kv_interleaved(kv_pool: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                          slot_mapping) -> np.ndarray:
    """A copy of the record pool with row i of k_new / v_new ([T][Hkv][D])
    written at slot slot_mapping[i] of the K and V members (negative = skip)."""
    bs = kv_pool.dtype["K"].shape[0]
    out = kv_pool.copy()
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        out[slot // bs]["K"][slot % bs] = k_new[i]
        out[slot // bs]["V"][slot % bs] = v_new[i]
    return out


def copy_blocks_interleaved(kv_pool: np.ndarray, pairs) -> np.ndarray:
    """A copy of the record pool with record dst := record src per pair
    (copy-on-write of the whole physical block)."""
    out = kv_pool.copy()
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        out[dst] = kv_pool[src]
    return out


def decode_attention_interleaved(q, kv_pool, block_table, seq_lens, scale, seqs=None):
    """Decode attention over a record pool: the two-pool attention with the
    records' K and V members as the pools."""
    k, v = split_kv_pool(kv_pool)
    return decode_attention(q, k, v, block_table, seq_lens, scale, seqs=seqs)


def decode_attention_interleaved_fp8(q, kv_pool, k_scale, v_scale, block_table, seq_lens, scale,
                                     seqs=None):
    """fp8 decode attention over a record pool of E4M3 bytes."""
    k, v = split_kv_pool(kv_pool)
    return decode_attention_fp8(q, k, v, k_scale, v_scale, block_table, seq_lens, scale,
                                seqs=seqs)
