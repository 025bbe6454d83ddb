"""fp16 byte-level reference for the two cache writes: append and block copy.

Test infrastructure only (see the package docstring).

* Append: the KV cache grows one token per decode step (lux-666 notes
  "PagedAttention", 问题从哪里来 / where the problem comes from; "Phase 7 ·
  Document 04 — PagedAttention", §2 primer). The step's new K/V row of a
  sequence goes to the pool slot the block manager assigned it; slot =
  physical_block * BS + offset, so it lands in block slot // BS at row
  slot % BS. A negative slot means "no write" for that row.
* Block copy: copy-on-write of a shared block (Document 04, §2 "block sharing
  (copy-on-write)": only the differing block is copied; lux-666 notes, prefix
  sharing copies at the copy-on-write boundary). The whole block, every row and
  head, is copied in both pools.
"""

from __future__ import annotations

import numpy as np


def append_kv(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray,
              v_new: np.ndarray, slot_mapping) -> tuple:
    """Return copies of the pools with row i of k_new/v_new at slot_mapping[i]."""
    BS = k_pool.shape[1]
    k = k_pool.copy()
    v = v_pool.copy()
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        k[slot // BS, slot % BS] = k_new[i]
        v[slot // BS, slot % BS] = v_new[i]
    return k, v


def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray, pairs) -> tuple:
    """Return copies of the pools with block dst := block src for each pair."""
    k = k_pool.copy()
    v = v_pool.copy()
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        k[dst] = k_pool[src]
        v[dst] = v_pool[src]
    return k, v


def swap_blocks(src_k: np.ndarray, src_v: np.ndarray, dst_k: np.ndarray, dst_v: np.ndarray,
                pairs) -> tuple:
    """Return copies of the destination pools with block dst := source block
    src for each (src, dst) pair: a block moving between the device pool and
    the host pool when a sequence is swapped out or back in (Document 04, §9:
    under memory pressure a sequence's blocks may be swapped)."""
    k = dst_k.copy()
    v = dst_v.copy()
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        k[dst] = src_k[src]
        v[dst] = src_v[src]
    return k, v
