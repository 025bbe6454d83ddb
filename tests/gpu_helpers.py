"""Shared helpers for the GPU parity tests: NaN poisoning of every pool row no
sequence may read, the attention tolerance, and oracle comparisons."""

from __future__ import annotations

import numpy as np

# |gpu - ref| <= ATOL + RTOL * |ref| elementwise (fp32 accumulate, fp16 out)
ATOL = 2e-3
RTOL = 1e-2


def assert_close_attention(gpu_fp16, ref_fp64, where=""):
    g = np.asarray(gpu_fp16, dtype=np.float64)
    r = np.asarray(ref_fp64, dtype=np.float64)
    assert g.shape == r.shape
    bad = ~(np.abs(g - r) <= ATOL + RTOL * np.abs(r))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.max(np.abs(g - r) - RTOL * np.abs(r))
        raise AssertionError(f"{where}: {int(bad.sum())} of {g.size} outside tolerance; "
                             f"first {idx.tolist()}; worst excess {worst:.3g}")


def used_rows_mask(tables, lens, nb, block_size):
    """[nb][block_size] bool: rows some sequence attends (t < len)."""
    keep = np.zeros((nb, block_size), dtype=bool)
    for row, L in zip(tables, lens):
        L = int(L)
        full, tail = divmod(L, block_size)
        if full:
            keep[np.asarray(row[:full], dtype=np.int64)] = True
        if tail:
            keep[int(row[full]), :tail] = True
    return keep


def poison_unread_rows(k_pool, v_pool, tables, lens, block_size):
    """Return copies of the pools where every row that no sequence attends
    (free blocks, and rows past each sequence's length in its last block)
    holds fp16 NaN. A kernel that reads outside the token set then produces
    NaN and fails the comparison."""
    keep = used_rows_mask(tables, lens, k_pool.shape[0], block_size)
    k = k_pool.copy()
    v = v_pool.copy()
    k[~keep] = np.float16(np.nan)
    v[~keep] = np.float16(np.nan)
    return k, v
