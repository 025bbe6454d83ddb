"""fp64 reference for single-query decode attention over a paged KV cache.

Test infrastructure only (see the package docstring).

What is computed, per sequence i and query head h:
    K_i[t], V_i[t] = pool[block_table[i][t // BS]][t % BS]   for t < L_i
    s_t  = scale * <q[i,h], K_i[t, kv(h)]>
    out  = sum_t softmax(s)_t * V_i[t, kv(h)]
The gather through the block table is the page-table indirection of
"Phase 7 · Document 04 — PagedAttention", §2 Core Concept ("the attention
kernel follows that indirection to gather K/V"; layout sketch `KVBlock` with
`K[BLOCK][HEADS][HEAD_DIM]` and `block_table[NUM_SEQS][MAX_BLOCKS]`), and of the
lux-666 notes "PagedAttention", 最小模型 (the kernel reads the block table and
visits physical blocks in logical token order).

Readings where the pages are silent:
  * K and V live in two separate pools, each [num_blocks][BS][H_kv][D]; the
    sketch's HEADS is the number of KV heads.
  * Grouped-query attention: query head h reads KV head h // G, G = Hq / Hkv
    (consecutive groups).
  * A sequence of length 0 attends to nothing; its output is all zeros.
  * The scale is a float32 value; it is widened exactly to fp64 here.
"""

from __future__ import annotations

import numpy as np


def gather_sequence(pool: np.ndarray, table_row, seq_len: int,
                    block_size: int) -> np.ndarray:
    """Rows 0..seq_len-1 of one sequence, in logical order, as fp64 [L][H][D].

    Logical token t sits in logical block t // BS at offset t % BS; the block
    table maps the logical block to its physical id in the pool.
    """
    L = int(seq_len)
    out = np.empty((L,) + tuple(pool.shape[2:]), dtype=np.float64)
    nblk = -(-L // block_size)
    for b in range(nblk):
        phys = int(table_row[b])
        lo = b * block_size
        hi = min(L, lo + block_size)
        out[lo:hi] = pool[phys, : hi - lo].astype(np.float64)
    return out


def _softmax_weighted_sum(s: np.ndarray, V: np.ndarray) -> np.ndarray:
    """sum_t softmax(s)_t V[t], with the max subtracted for stability."""
    e = np.exp(s - s.max())
    return (e / e.sum()) @ V


def decode_attention_one(q_row: np.ndarray, K: np.ndarray, V: np.ndarray,
                         scale: float) -> np.ndarray:
    """Attention of one query vector over contiguous K [L][D], V [L][D] (fp64)."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[-1], dtype=np.float64)
    s = float(scale) * (K @ q_row.astype(np.float64))
    return _softmax_weighted_sum(s, V)


def decode_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                     block_table: np.ndarray, seq_lens, scale,
                     seqs=None, heads=None) -> np.ndarray:
    """Paged decode attention, fp64 result [S][Hq][D].

    q [S][Hq][D]; k_pool, v_pool [NB][BS][Hkv][D]; block_table int [S][MB];
    seq_lens [S] (tokens attended, the appended one included); scale fp32.
    `seqs` / `heads` restrict the work to a sample (other rows stay zero).
    """
    S, Hq, D = q.shape
    BS = k_pool.shape[1]
    Hkv = k_pool.shape[2]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    G = Hq // Hkv
    sc = float(np.float32(scale))
    out = np.zeros((S, Hq, D), dtype=np.float64)
    seq_iter = range(S) if seqs is None else seqs
    for i in seq_iter:
        L = int(seq_lens[i])
        if L == 0:
            continue
        K = gather_sequence(k_pool, block_table[i], L, BS)
        V = gather_sequence(v_pool, block_table[i], L, BS)
        for h in (range(Hq) if heads is None else heads):
            kv = h // G
            out[i, h] = decode_attention_one(q[i, h], K[:, kv, :], V[:, kv, :], sc)
    return out


# --- split-context form -----------------------------------------------------
# Not on the pages: the split-context (flash-decoding) partition + merge is the
# method's way to spread one long sequence over many workers. It must give the
# same result as the unsplit definition above; these functions state the
# partition and the log-sum-exp merge so that identity can be tested.

def split_partials(s: np.ndarray, V: np.ndarray, bounds):
    """Per-chunk partials of softmax attention.

    For each chunk [a, b): m = max s[a:b], l = sum exp(s[a:b] - m),
    acc = sum exp(s[a:b] - m) V[a:b]. Empty chunks give m = -inf, l = 0, acc = 0.
    """
    ms, ls, accs = [], [], []
    for a, b in bounds:
        if b <= a:
            ms.append(-np.inf)
            ls.append(0.0)
            accs.append(np.zeros(V.shape[-1]))
            continue
        m = s[a:b].max()
        e = np.exp(s[a:b] - m)
        ms.append(m)
        ls.append(e.sum())
        accs.append(e @ V[a:b])
    return np.array(ms), np.array(ls), np.array(accs)


def merge_partials(ms, ls, accs) -> np.ndarray:
    """Combine chunk partials: M = max m_j, w_j = exp(m_j - M),
    out = sum_j w_j acc_j / sum_j w_j l_j."""
    ms = np.asarray(ms, dtype=np.float64)
    M = ms.max()
    if not np.isfinite(M):
        return np.zeros(np.asarray(accs).shape[-1])
    w = np.exp(ms - M)
    return (w[:, None] * np.asarray(accs)).sum(0) / (w * np.asarray(ls)).sum()


def split_context_attention(q_row, K, V, scale, chunk: int) -> np.ndarray:
    """Attention of one query computed chunk by chunk and merged."""
    L = K.shape[0]
    if L == 0:
        return np.zeros(V.shape[-1])
    s = float(scale) * (K @ q_row.astype(np.float64))
    bounds = [(a, min(L, a + chunk)) for a in range(0, L, chunk)]
    return merge_partials(*split_partials(s, V, bounds))
