"""paged_kv_cache_40_gb300 — paged decode attention for GB300 behind a C ABI.

This module is the thin Python face of libpa.so (include/pa.h): each function
has the C name, checks and marshals torch tensors (device pointers, sizes, the
current CUDA stream) and calls the library. All device work runs in libpa's
CUDA kernels; nothing here computes on the host, and there is no fallback.

Device calls                            Host block manager
  pa_append_kv, pa_append_kv_fp8          BlockAllocator (pa_alloc_*), with
  pa_copy_blocks, pa_copy_blocks_fp8      a host pool for swapping
  pa_swap_blocks
  pa_decode_attention (+ _fp8, _shared_prefix, _fixed_scratch)
  pa_decode_append_attention: the append and the attention in one kernel
  pa_decode_workspace_bytes / _init
  pa_device_error

Pools are [num_blocks][block_size][kv_heads][head_dim] tensors, dense or the
K and V member views of one record pool (kv_block_pool / kv_views); the block
stride is read from the tensors. Attention outputs may be pinned host memory.
"""

from __future__ import annotations

import ctypes
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

from ._lib import (  # noqa: F401
    AllocStats,
    OutOfBlocksError,
    PaError,
    PA_DEVERR_BAD_BLOCK,
    PA_DEVERR_BAD_LEN,
    PA_DEVERR_BAD_SLOT,
    PA_DEVERR_TIMEOUT,
    LIB_PATH,
    check as _check,
    load as _load,
)

__all__ = [
    "pa_append_kv", "pa_copy_blocks", "pa_decode_attention", "pa_decode_append_attention",
    "pa_decode_workspace_bytes", "pa_decode_workspace_init", "pa_device_error",
    "pa_append_kv_fp8", "pa_copy_blocks_fp8", "pa_decode_attention_fp8",
    "pa_decode_attention_shared_prefix", "pa_decode_shared_prefix_workspace_bytes",
    "pa_swap_blocks",
    "pa_decode_attention_fixed_scratch", "kv_block_pool", "kv_views",
    "pa_version", "pa_kernel_launches", "pa_set_wait_limit_ns", "BlockAllocator", "PaError",
    "OutOfBlocksError", "lib",
]


def lib() -> ctypes.CDLL:
    return _load()


def pa_version() -> int:
    return int(_load().pa_version())


def pa_kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far (a monotonic
    count; read it before and after a region of calls)."""
    return int(_load().pa_kernel_launches())


# ----------------------------------------------------------------- helpers --
def _torch():
    import torch
    return torch


def _stream_ptr(stream) -> ctypes.c_void_p:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _dev(t, name, dtype, ndim=None, host_ok=False):
    """Pointer of a contiguous tensor the kernels use: a CUDA tensor, or (for
    the arrays a call reads or writes in place, host_ok) pinned host memory,
    which the kernels reach through its device mapping."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" +
                         (" or pinned host memory" if host_ok else ""))
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _in(t, name, dtype):
    return _dev(t, name, dtype, host_ok=True)


def _out(t, like):
    """Output pointer: a CUDA tensor, or pinned host memory that the kernel
    writes through its device mapping (no copy back)."""
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float16 or not t.is_contiguous():
        raise TypeError("out must be a contiguous float16 tensor")
    if tuple(t.shape) != tuple(like.shape):
        raise ValueError("out must have q's shape")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("out must be a CUDA tensor or pinned host memory")
    return ctypes.c_void_p(t.data_ptr())


def _block_stride(t, name) -> int:
    """Values from one block of a pool to the next; each block itself must be
    a contiguous [block_size][kv_heads][head_dim] array."""
    nb, bs, hkv, d = (int(x) for x in t.shape)
    if (bs > 1 and t.stride(1) != hkv * d) or (hkv > 1 and t.stride(2) != d) or \
            (d > 1 and t.stride(3) != 1):
        raise ValueError(f"{name}: each block must be a contiguous [block_size][kv_heads][head_dim]")
    return int(t.stride(0)) if nb > 1 else bs * hkv * d


def _pool_dims(k_pool, v_pool):
    """(num_blocks, block_size, kv_heads, head_dim, block stride in values) of
    a K/V pool pair: two dense pools, or the two member views of one record
    pool (kv_block_pool)."""
    if k_pool.dim() != 4 or tuple(k_pool.shape) != tuple(v_pool.shape):
        raise ValueError("k_pool and v_pool must both be [num_blocks][block_size][kv_heads][head_dim]")
    nb, bs, hkv, d = (int(x) for x in k_pool.shape)
    stride = _block_stride(k_pool, "k_pool")
    if _block_stride(v_pool, "v_pool") != stride:
        raise ValueError("k_pool and v_pool must have the same block stride")
    return nb, bs, hkv, d, stride


def _pool(t, name, dtype):
    """Device pointer of a pool (blocks may be strided; see _block_stride)."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libpa has no host path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def kv_block_pool(num_blocks, block_size, num_kv_heads, head_dim, dtype=None, device=None):
    """One pool of per-block records, each a block's K rows followed by its V
    rows (the layout sketch of "Phase 7 · Document 04 — PagedAttention", §2):
    a zero-filled tensor [num_blocks][2][block_size][num_kv_heads][head_dim]
    (fp16 by default; torch.uint8 for an E4M3 cache). kv_views() gives the K
    and V pools every call takes."""
    torch = _torch()
    return torch.zeros((num_blocks, 2, block_size, num_kv_heads, head_dim),
                       dtype=dtype or torch.float16, device=device or "cuda")


def kv_views(kv_pool):
    """(k_pool, v_pool) views [NB][BS][Hkv][D] of a record pool (kv_block_pool);
    consecutive blocks of each are two blocks apart."""
    if kv_pool.dim() != 5 or int(kv_pool.shape[1]) != 2:
        raise ValueError("kv_pool must be [num_blocks][2][block_size][kv_heads][head_dim]")
    return kv_pool[:, 0], kv_pool[:, 1]


# ------------------------------------------------------------ device calls --
def pa_append_kv(k_new, v_new, k_pool, v_pool, slot_mapping, stream=None) -> None:
    """Write row i of k_new/v_new ([T][Hkv][D] fp16) into pool slot
    slot_mapping[i] (int32; negative = skip)."""
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    T = int(slot_mapping.numel())
    if tuple(k_new.shape) != (T, hkv, d) or tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("k_new/v_new must be [num_tokens][kv_heads][head_dim]")
    args = (_in(k_new, "k_new", torch.float16), _in(v_new, "v_new", torch.float16),
            _pool(k_pool, "k_pool", torch.float16), _pool(v_pool, "v_pool", torch.float16),
            _in(slot_mapping, "slot_mapping", torch.int32))
    _check(_load().pa_append_kv(*args, T, hkv, d, bs, nb, stride, _stream_ptr(stream)))


def pa_copy_blocks(k_pool, v_pool, pairs, stream=None) -> None:
    """Copy block src to block dst in both pools for each (src, dst) row of
    pairs (int32 [n][2])."""
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [n][2]")
    n = int(pairs.shape[0])
    args = (_pool(k_pool, "k_pool", torch.float16), _pool(v_pool, "v_pool", torch.float16),
            _in(pairs, "pairs", torch.int32))
    _check(_load().pa_copy_blocks(*args, n, hkv, d, bs, nb, stride, _stream_ptr(stream)))


def pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                              block_size, max_blocks_per_seq,
                              partition_tokens: int = 0) -> int:
    n = int(_load().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              block_size, max_blocks_per_seq, partition_tokens))
    if n == 0 and num_seqs > 0:
        raise PaError(1, "pa_decode_workspace_bytes: unsupported or invalid shape")
    return n


def pa_decode_workspace_init(workspace, num_seqs, num_kv_heads, stream=None) -> None:
    torch = _torch()
    ptr = _dev(workspace, "workspace", torch.uint8)
    _check(_load().pa_decode_workspace_init(ptr, workspace.numel(), num_seqs, num_kv_heads,
                                            _stream_ptr(stream)))


def alloc_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                    max_blocks_per_seq, partition_tokens: int = 0, device=None):
    """A zero-filled uint8 CUDA buffer sized for pa_decode_attention."""
    torch = _torch()
    n = pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                  max_blocks_per_seq, partition_tokens)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def pa_decode_attention(q, k_pool, v_pool, block_table, seq_lens, scale, out=None,
                        workspace=None, partition_tokens: int = 0, stream=None):
    """Paged decode attention. q [S][Hq][D] fp16; pools [NB][BS][Hkv][D] fp16;
    block_table int32 [S][MB]; seq_lens int32 [S]. Returns out [S][Hq][D] fp16."""
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    if q.dim() != 3 or int(q.shape[2]) != d:
        raise ValueError("q must be [num_seqs][num_q_heads][head_dim]")
    S, hq = int(q.shape[0]), int(q.shape[1])
    if block_table.dim() != 2 or int(block_table.shape[0]) != S:
        raise ValueError("block_table must be [num_seqs][max_blocks_per_seq]")
    mb = int(block_table.shape[1])
    if tuple(seq_lens.shape) != (S,):
        raise ValueError("seq_lens must be [num_seqs]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float16, device=k_pool.device)
    if workspace is None:
        workspace = alloc_workspace(S, hq, hkv, d, bs, mb, partition_tokens, k_pool.device)
    args = (_in(q, "q", torch.float16), _pool(k_pool, "k_pool", torch.float16),
            _pool(v_pool, "v_pool", torch.float16), _in(block_table, "block_table", torch.int32),
            _in(seq_lens, "seq_lens", torch.int32))
    _check(_load().pa_decode_attention(
        *args, S, hq, hkv, d, bs, mb, nb, stride, ctypes.c_float(float(scale)),
        _out(out, q), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), partition_tokens, _stream_ptr(stream)))
    return out


def pa_decode_append_attention(q, k_new, v_new, slot_mapping, k_pool, v_pool, block_table,
                               seq_lens, scale, out=None, workspace=None,
                               partition_tokens: int = 0, stream=None):
    """pa_append_kv then pa_decode_attention in one kernel, one new token per
    sequence (k_new/v_new [S][Hkv][D] fp16, row i for sequence i;
    slot_mapping int32 [S], the row of each sequence's last token). The
    other arguments are pa_decode_attention's. Returns out."""
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    if q.dim() != 3 or int(q.shape[2]) != d:
        raise ValueError("q must be [num_seqs][num_q_heads][head_dim]")
    S, hq = int(q.shape[0]), int(q.shape[1])
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        if tuple(t.shape) != (S, hkv, d):
            raise ValueError(f"{name} must be [num_seqs][num_kv_heads][head_dim]")
    if tuple(slot_mapping.shape) != (S,):
        raise ValueError("slot_mapping must be [num_seqs]")
    if block_table.dim() != 2 or int(block_table.shape[0]) != S:
        raise ValueError("block_table must be [num_seqs][max_blocks_per_seq]")
    mb = int(block_table.shape[1])
    if tuple(seq_lens.shape) != (S,):
        raise ValueError("seq_lens must be [num_seqs]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float16, device=k_pool.device)
    if workspace is None:
        workspace = alloc_workspace(S, hq, hkv, d, bs, mb, partition_tokens, k_pool.device)
    _check(_load().pa_decode_append_attention(
        _in(q, "q", torch.float16), _in(k_new, "k_new", torch.float16),
        _in(v_new, "v_new", torch.float16), _in(slot_mapping, "slot_mapping", torch.int32),
        _pool(k_pool, "k_pool", torch.float16), _pool(v_pool, "v_pool", torch.float16),
        _in(block_table, "block_table", torch.int32), _in(seq_lens, "seq_lens", torch.int32),
        S, hq, hkv, d, bs, mb, nb, stride, ctypes.c_float(float(scale)), _out(out, q),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), partition_tokens,
        _stream_ptr(stream)))
    return out


# ------------------------------------------------------------------ swapping --
def pa_swap_blocks(src_k, src_v, dst_k, dst_v, pairs, stream=None) -> None:
    """Block pairs[i][1] of dst := block pairs[i][0] of src, for K and V. Pools
    are [blocks][BS][Hkv][D] of one element type (dense, or the member views
    of a record pool), each a CUDA tensor or pinned CPU memory; pairs is int32
    [n][2], CUDA or pinned CPU. With src_v and dst_v None, src_k and dst_k are
    record pools (kv_block_pool layout) and whole records move."""
    torch = _torch()
    records = src_v is None and dst_v is None
    if (src_v is None) != (dst_v is None):
        raise ValueError("src_v and dst_v must both be tensors or both None")
    named = [(src_k, "src_k"), (dst_k, "dst_k"), (pairs, "pairs")]
    if not records:
        named += [(src_v, "src_v"), (dst_v, "dst_v")]
    for t, name in named:
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{name} must be a tensor")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if src_k.shape[1:] != dst_k.shape[1:] or src_k.dtype != dst_k.dtype:
        raise ValueError("source and destination pools must share their block shape and type")
    if pairs.dtype != torch.int32 or pairs.dim() != 2 or pairs.shape[1] != 2 or \
            not pairs.is_contiguous():
        raise ValueError("pairs must be contiguous int32 [n][2]")
    esz = src_k.element_size()
    if records:
        if src_k.dim() != 5 or int(src_k.shape[1]) != 2:
            raise ValueError("record pools must be [blocks][2][block_size][kv_heads][head_dim]")
        for t, name in ((src_k, "src_k"), (dst_k, "dst_k")):
            if not t[0].is_contiguous():
                raise ValueError(f"{name}: each record must be contiguous")
        s_stride = int(src_k.stride(0)) if src_k.shape[0] > 1 else int(src_k[0].numel())
        d_stride = int(dst_k.stride(0)) if dst_k.shape[0] > 1 else int(dst_k[0].numel())
        sv = dv = ctypes.c_void_p(0)
    else:
        if src_k.dim() != 4 or src_k.shape != src_v.shape or dst_k.shape != dst_v.shape or \
                src_v.dtype != src_k.dtype or dst_v.dtype != dst_k.dtype:
            raise ValueError("source and destination pools must share their block shape and type")
        s_stride = _block_stride(src_k, "src_k")
        d_stride = _block_stride(dst_k, "dst_k")
        if _block_stride(src_v, "src_v") != s_stride or _block_stride(dst_v, "dst_v") != d_stride:
            raise ValueError("the K and V pools of one side must have the same block stride")
        sv, dv = ctypes.c_void_p(src_v.data_ptr()), ctypes.c_void_p(dst_v.data_ptr())
    block_bytes = int(src_k[0].numel() * esz)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    _check(_load().pa_swap_blocks(ptr(src_k), sv, int(src_k.shape[0]), s_stride * esz,
                                  ptr(dst_k), dv, int(dst_k.shape[0]), d_stride * esz,
                                  ptr(pairs), int(pairs.shape[0]), block_bytes,
                                  _stream_ptr(stream)))


# ------------------------------------------------------------ shared prefix --
def pa_decode_shared_prefix_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                            block_size, max_blocks_per_seq,
                                            num_prefix_blocks) -> int:
    n = int(_load().pa_decode_shared_prefix_workspace_bytes(
        num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
        num_prefix_blocks))
    if n == 0 and num_seqs > 0:
        raise PaError(1, "pa_decode_shared_prefix_workspace_bytes: unsupported or invalid shape")
    return n


def pa_decode_attention_shared_prefix(q, k_pool, v_pool, prefix_blocks, block_table, seq_lens,
                                      scale, out=None, workspace=None, stream=None):
    """pa_decode_attention for sequences that all begin with the physical
    blocks `prefix_blocks` (int32 [P]): block_table[i][:P] must equal them and
    seq_lens[i] >= P * block_size. The prefix blocks are read once for the
    whole batch. Returns out [S][Hq][D] fp16."""
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    if q.dim() != 3 or int(q.shape[2]) != d:
        raise ValueError("q must be [num_seqs][num_q_heads][head_dim]")
    S, hq = int(q.shape[0]), int(q.shape[1])
    if block_table.dim() != 2 or int(block_table.shape[0]) != S:
        raise ValueError("block_table must be [num_seqs][max_blocks_per_seq]")
    mb = int(block_table.shape[1])
    if tuple(seq_lens.shape) != (S,) or prefix_blocks.dim() != 1:
        raise ValueError("seq_lens must be [num_seqs] and prefix_blocks one-dimensional")
    P = int(prefix_blocks.numel())
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float16, device=k_pool.device)
    if workspace is None:
        n = pa_decode_shared_prefix_workspace_bytes(S, hq, hkv, d, bs, mb, P)
        workspace = torch.zeros(max(n, 16), dtype=torch.uint8, device=k_pool.device)
    args = (_in(q, "q", torch.float16), _pool(k_pool, "k_pool", torch.float16),
            _pool(v_pool, "v_pool", torch.float16),
            _in(prefix_blocks, "prefix_blocks", torch.int32) if P else ctypes.c_void_p(0), P,
            _in(block_table, "block_table", torch.int32),
            _in(seq_lens, "seq_lens", torch.int32))
    _check(_load().pa_decode_attention_shared_prefix(
        *args, S, hq, hkv, d, bs, mb, nb, stride, ctypes.c_float(float(scale)),
        _out(out, q), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream_ptr(stream)))
    return out


# ------------------------------------------------------- fp8 (E4M3) cache --
def _scales(k_scale, v_scale, hkv):
    torch = _torch()
    if tuple(k_scale.shape) != (hkv,) or tuple(v_scale.shape) != (hkv,):
        raise ValueError("k_scale and v_scale must be [num_kv_heads] fp32")
    return _in(k_scale, "k_scale", torch.float32), _in(v_scale, "v_scale", torch.float32)


def pa_append_kv_fp8(k_new, v_new, k_pool, v_pool, slot_mapping, k_scale, v_scale,
                     stream=None) -> None:
    """pa_append_kv into E4M3 pools (uint8 [NB][BS][Hkv][D]): row i of
    k_new/v_new (fp16 [T][Hkv][D]) is quantized with the per-KV-head scales
    and written at slot slot_mapping[i]."""
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    T = int(slot_mapping.numel())
    if tuple(k_new.shape) != (T, hkv, d) or tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("k_new/v_new must be [num_tokens][kv_heads][head_dim]")
    ks, vs = _scales(k_scale, v_scale, hkv)
    args = (_in(k_new, "k_new", torch.float16), _in(v_new, "v_new", torch.float16),
            _pool(k_pool, "k_pool", torch.uint8), _pool(v_pool, "v_pool", torch.uint8),
            _in(slot_mapping, "slot_mapping", torch.int32), ks, vs)
    _check(_load().pa_append_kv_fp8(*args, T, hkv, d, bs, nb, stride, _stream_ptr(stream)))


def pa_copy_blocks_fp8(k_pool, v_pool, pairs, stream=None) -> None:
    """pa_copy_blocks over E4M3 pools (uint8 [NB][BS][Hkv][D])."""
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [n][2]")
    n = int(pairs.shape[0])
    args = (_pool(k_pool, "k_pool", torch.uint8), _pool(v_pool, "v_pool", torch.uint8),
            _in(pairs, "pairs", torch.int32))
    _check(_load().pa_copy_blocks_fp8(*args, n, hkv, d, bs, nb, stride, _stream_ptr(stream)))


def pa_decode_attention_fp8(q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, scale,
                            out=None, workspace=None, partition_tokens: int = 0, stream=None):
    """pa_decode_attention over E4M3 pools (uint8 [NB][BS][Hkv][D]) with fp32
    per-KV-head scales k_scale, v_scale [Hkv]. Returns out [S][Hq][D] fp16."""
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    if q.dim() != 3 or int(q.shape[2]) != d:
        raise ValueError("q must be [num_seqs][num_q_heads][head_dim]")
    S, hq = int(q.shape[0]), int(q.shape[1])
    if block_table.dim() != 2 or int(block_table.shape[0]) != S:
        raise ValueError("block_table must be [num_seqs][max_blocks_per_seq]")
    mb = int(block_table.shape[1])
    if tuple(seq_lens.shape) != (S,):
        raise ValueError("seq_lens must be [num_seqs]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float16, device=k_pool.device)
    if workspace is None:
        workspace = alloc_workspace(S, hq, hkv, d, bs, mb, partition_tokens, k_pool.device)
    ks, vs = _scales(k_scale, v_scale, hkv)
    args = (_in(q, "q", torch.float16), _pool(k_pool, "k_pool", torch.uint8),
            _pool(v_pool, "v_pool", torch.uint8), ks, vs,
            _in(block_table, "block_table", torch.int32),
            _in(seq_lens, "seq_lens", torch.int32))
    _check(_load().pa_decode_attention_fp8(
        *args, S, hq, hkv, d, bs, mb, nb, stride, ctypes.c_float(float(scale)),
        _out(out, q), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), partition_tokens, _stream_ptr(stream)))
    return out


def pa_decode_attention_fixed_scratch(q, k_pool, v_pool, block_table, seq_lens, scale,
                                      out=None, partition_tokens: int = 0, stream=None):
    """pa_decode_attention for callers that cannot provide a workspace.

    For a process that cannot allocate device memory on the decode path (all
    of it already belongs to its own KV pool and allocator, or cudaMalloc's
    device synchronisation is not acceptable there): the scratch is a fixed
    16 MiB array inside libpa. Same inputs and result as pa_decode_attention;
    shapes needing more scratch raise PaError (PA_ERR_UNSUPPORTED). Calls that
    overlap on the GPU share that array and must not be issued.
    """
    torch = _torch()
    nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
    if q.dim() != 3 or int(q.shape[2]) != d:
        raise ValueError("q must be [num_seqs][num_q_heads][head_dim]")
    S, hq = int(q.shape[0]), int(q.shape[1])
    if block_table.dim() != 2 or int(block_table.shape[0]) != S:
        raise ValueError("block_table must be [num_seqs][max_blocks_per_seq]")
    if tuple(seq_lens.shape) != (S,):
        raise ValueError("seq_lens must be [num_seqs]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float16, device=k_pool.device)
    args = (_in(q, "q", torch.float16), _pool(k_pool, "k_pool", torch.float16),
            _pool(v_pool, "v_pool", torch.float16), _in(block_table, "block_table", torch.int32),
            _in(seq_lens, "seq_lens", torch.int32))
    _check(_load().pa_decode_attention_fixed_scratch(
        *args, S, hq, hkv, d, bs, int(block_table.shape[1]), nb, stride,
        ctypes.c_float(float(scale)),
        _out(out, q), partition_tokens, _stream_ptr(stream)))
    return out


class PreparedDecodeStep:
    """pa_decode_step with its arguments marshalled once: the block manager
    plans each call's step into `plan` (slots [n], copy-on-write pairs
    [n][2], table [n][max_blocks], lengths [n]: pinned int32 host tensors
    that the kernels read in place), then the copies, the append and the
    attention are enqueued on `stream`, all in one library call. The
    tensors are fixed for the object's life; each call returns the number of
    copy-on-write pairs it planned."""

    def __init__(self, alloc, seq_ids, max_blocks, plan, q, k_new, v_new, k_pool, v_pool, scale,
                 out, workspace, partition_tokens: int = 0, stream=None, k_scale=None,
                 v_scale=None):
        """With uint8 pools (E4M3 codes) and device fp32 k_scale / v_scale
        [num_kv_heads] the step is pa_decode_step_fp8."""
        torch = _torch()
        fp8 = k_pool.dtype == torch.uint8
        if fp8 and (k_scale is None or v_scale is None):
            raise ValueError("an E4M3 cache needs k_scale and v_scale")
        nb, bs, hkv, d, stride = _pool_dims(k_pool, v_pool)
        if bs != alloc.block_size or nb != alloc.num_blocks:
            raise ValueError("the pools and the block manager differ in block size or blocks")
        self.seq_ids = np.ascontiguousarray(seq_ids, dtype=np.int64).reshape(-1)
        n = int(self.seq_ids.size)
        slots, pairs, table, lens = plan
        for t, shape, name in ((slots, (n,), "slots"), (pairs, (n, 2), "pairs"),
                               (table, (n, max_blocks), "table"), (lens, (n,), "lens")):
            if t.is_cuda or not t.is_pinned() or t.dtype != torch.int32 or \
                    not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError(f"plan {name} must be a pinned int32 host tensor of shape {shape}")
        if q.dim() != 3 or int(q.shape[0]) != n or int(q.shape[2]) != d:
            raise ValueError("q must be [num_seqs][num_q_heads][head_dim]")
        hq = int(q.shape[1])
        self.plan = plan
        self._keep = (alloc, q, k_new, v_new, k_pool, v_pool, out, workspace, k_scale, v_scale)
        self._ncow = ctypes.c_int()
        ids = self.seq_ids if n else np.zeros(1, np.int64)
        self._ids = ids
        head = (alloc._h, ids.ctypes.data, n, max_blocks,
                ctypes.c_void_p(slots.data_ptr()), ctypes.c_void_p(pairs.data_ptr()),
                ctypes.c_void_p(table.data_ptr()), ctypes.c_void_p(lens.data_ptr()),
                ctypes.byref(self._ncow), _in(q, "q", torch.float16),
                _in(k_new, "k_new", torch.float16), _in(v_new, "v_new", torch.float16))
        tail = (hq, hkv, d, nb, stride, ctypes.c_float(float(scale)), _out(out, q),
                _dev(workspace, "workspace", torch.uint8), workspace.numel(),
                partition_tokens, _stream_ptr(stream))
        if fp8:
            self._fn = _load().pa_decode_step_fp8
            self._args = head + (_pool(k_pool, "k_pool", torch.uint8),
                                 _pool(v_pool, "v_pool", torch.uint8),
                                 _dev(k_scale, "k_scale", torch.float32),
                                 _dev(v_scale, "v_scale", torch.float32)) + tail
        else:
            self._fn = _load().pa_decode_step
            self._args = head + (_pool(k_pool, "k_pool", torch.float16),
                                 _pool(v_pool, "v_pool", torch.float16)) + tail

    def __call__(self) -> int:
        _check(self._fn(*self._args))
        return self._ncow.value


def pa_device_error(stream=None) -> int:
    """Read and clear the device error word (synchronises the stream).
    Returns the PA_DEVERR_* bit set; raises PaError if any bit was set."""
    flags = ctypes.c_int32(0)
    st = _load().pa_device_error(_stream_ptr(stream), ctypes.byref(flags))
    if st != 0:
        err = PaError(st, _load().pa_last_error().decode(errors="replace"))
        err.flags = int(flags.value)
        raise err
    return int(flags.value)


def pa_set_wait_limit_ns(limit_ns: int) -> None:
    """Time limit of the attention kernels' pipeline waits for later calls
    (0 restores the default of about one second). A wait that runs out sets
    PA_DEVERR_TIMEOUT and the launch's outputs are undefined; tests use a
    short limit to run that path."""
    _check(_load().pa_set_wait_limit_ns(int(limit_ns)))


# ------------------------------------------------------------ host allocator --
def _i32_array(values):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr


def _i64_ids(seqs) -> "np.ndarray":
    """Sequence ids as a contiguous int64 buffer (at least one element, so
    that its address is valid even for an empty batch)."""
    ids = np.ascontiguousarray(seqs, dtype=np.int64).reshape(-1)
    return ids if ids.size else np.zeros(1, np.int64)


class BlockAllocator:
    """The host block manager of libpa (pa_alloc_*), one handle per pool."""

    def __init__(self, num_blocks: int, block_size: int,
                 initial_free_order: Optional[Sequence[int]] = None):
        L = _load()
        handle = ctypes.c_void_p()
        order = None
        if initial_free_order is not None:
            if len(initial_free_order) != num_blocks:
                raise ValueError("initial free order must list every block")
            order = _i32_array(list(initial_free_order))
        _check(L.pa_alloc_create(num_blocks, block_size, order, ctypes.byref(handle)))
        self._h = handle
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if getattr(self, "_h", None) and self._h.value:
            _load().pa_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq: int, length: int) -> None:
        _check(_load().pa_alloc_add_seq(self._h, seq, length))

    def fork(self, parent: int, child: int) -> None:
        _check(_load().pa_alloc_fork(self._h, parent, child))

    def append_slot(self, seq: int) -> Tuple[int, int, int]:
        s, a, b = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(_load().pa_alloc_append_slot(self._h, seq, ctypes.byref(s), ctypes.byref(a),
                                            ctypes.byref(b)))
        return s.value, a.value, b.value

    def append_slots(self, seqs: Sequence[int]):
        """One decode step: (slots int32 list, cow pairs list of (src, dst))."""
        ids = _i64_ids(seqs)
        n = len(seqs)
        slots = np.empty(max(n, 1), np.int32)
        pairs = np.empty(max(2 * n, 2), np.int32)
        ncow, ndone = ctypes.c_int(), ctypes.c_int()
        _check(_load().pa_alloc_append_slots(self._h, ids.ctypes.data, n, slots.ctypes.data,
                                             pairs.ctypes.data, ctypes.byref(ncow),
                                             ctypes.byref(ndone)))
        return slots[:n].tolist(), list(map(tuple, pairs[:2 * ncow.value].reshape(-1, 2).tolist()))

    def plan_step(self, seqs: Sequence[int], max_blocks: int, fill: int = -1, out=None):
        """One decode step of the batch `seqs` in one library call
        (pa_alloc_plan_step): (slots int32 [n], copy-on-write pairs int32
        [ncow][2], table int32 [n][max_blocks], seq_lens int32 [n]) after the
        appends. `out` = (slots, pairs, table, lens) preallocated contiguous
        int32 numpy arrays of shapes [n], [n][2], [n][max_blocks], [n] (for
        instance views of pinned host memory the kernels read) to be written
        in place; the returned pairs are then a view of the first ncow rows."""
        ids = _i64_ids(seqs)
        n = len(seqs)
        if out is None:
            out = (np.empty(max(n, 1), np.int32), np.empty((max(n, 1), 2), np.int32),
                   np.empty((max(n, 1), max_blocks), np.int32), np.empty(max(n, 1), np.int32))
        slots, pairs, table, lens = out
        for arr, need in ((slots, n), (pairs, 2 * n), (table, n * max_blocks), (lens, n)):
            if arr.dtype != np.int32 or not arr.flags.c_contiguous or arr.size < need:
                raise ValueError("plan_step outputs must be contiguous int32 arrays of "
                                 "[n], [n][2], [n][max_blocks], [n]")
        ncow = ctypes.c_int()
        _check(_load().pa_alloc_plan_step(self._h, ids.ctypes.data, n, max_blocks, fill,
                                          slots.ctypes.data, pairs.ctypes.data,
                                          ctypes.byref(ncow), table.ctypes.data,
                                          lens.ctypes.data))
        return (slots[:n], pairs.reshape(-1, 2)[:ncow.value],
                table.reshape(-1, max_blocks)[:n], lens[:n])

    def free_seq(self, seq: int) -> None:
        _check(_load().pa_alloc_free_seq(self._h, seq))

    def table(self, seq: int):
        n = ctypes.c_int()
        st = _load().pa_alloc_get_table(self._h, seq, None, 0, ctypes.byref(n))
        if st not in (0, 1):
            _check(st)
        buf = (ctypes.c_int32 * max(n.value, 1))()
        _check(_load().pa_alloc_get_table(self._h, seq, buf, n.value, ctypes.byref(n)))
        return list(buf[:n.value])

    def seq_len(self, seq: int) -> int:
        v = ctypes.c_int64()
        _check(_load().pa_alloc_seq_len(self._h, seq, ctypes.byref(v)))
        return v.value

    def build_tables(self, seqs: Sequence[int], max_blocks: int, fill: int = -1):
        """(table int32 numpy [n][max_blocks], seq_lens int32 numpy [n])."""
        ids = _i64_ids(seqs)
        n = len(seqs)
        table = np.empty((max(n, 1), max_blocks), dtype=np.int32)
        lens = np.empty((max(n, 1),), dtype=np.int32)
        _check(_load().pa_alloc_build_tables(self._h, ids.ctypes.data, n, max_blocks, fill,
                                             table.ctypes.data, lens.ctypes.data))
        return table[:n], lens[:n]

    def shared_prefix(self, seqs: Sequence[int]):
        """int32 numpy array of the whole blocks every sequence of `seqs`
        begins with (pa_alloc_shared_prefix): the prefix that
        pa_decode_attention_shared_prefix takes for this batch."""
        ids = _i64_ids(seqs)
        cap = max(self.num_blocks, 1)
        out = np.empty(cap, np.int32)
        k = ctypes.c_int()
        _check(_load().pa_alloc_shared_prefix(self._h, ids.ctypes.data, len(seqs),
                                              out.ctypes.data, cap, ctypes.byref(k)))
        return out[:k.value].copy()

    def stats(self) -> dict:
        st = AllocStats()
        _check(_load().pa_alloc_stats(self._h, ctypes.byref(st)))
        return {
            "num_blocks": st.num_blocks, "free": st.free_blocks, "used": st.used_blocks,
            "shared": st.shared_blocks, "cow_copies": st.cow_copies,
            "alloc_failures": st.alloc_failures, "total_refs": st.total_refs,
            "num_seqs": st.num_seqs,
        }

    # -- swapping -------------------------------------------------------------
    def add_host_pool(self, num_host_blocks: int, initial_free_order=None) -> None:
        order = None
        if initial_free_order is not None:
            order = _i32_array(initial_free_order)
        _check(_load().pa_alloc_add_host_pool(self._h, int(num_host_blocks), order))
        self.num_host_blocks = int(num_host_blocks)

    def _swap(self, fn, seq):
        # a sequence never holds more blocks than either pool
        cap = max(self.num_blocks, getattr(self, "num_host_blocks", 0), 1)
        n = ctypes.c_int()
        buf = (ctypes.c_int32 * (2 * cap))()
        _check(fn(self._h, seq, buf, cap, ctypes.byref(n)))
        return [(buf[2 * i], buf[2 * i + 1]) for i in range(n.value)]

    def swap_out(self, seq: int):
        """Move the sequence to host blocks: (device, host) pairs to copy."""
        return self._swap(_load().pa_alloc_swap_out, seq)

    def swap_in(self, seq: int):
        """Bring the sequence back to fresh device blocks: (host, device) pairs."""
        return self._swap(_load().pa_alloc_swap_in, seq)

    def export_host_state(self):
        """(host free list front to back, swapped-out sequences, swap-outs,
        swap-ins)."""
        nh = getattr(self, "num_host_blocks", 0)
        fo = (ctypes.c_int32 * max(nh, 1))()
        nf = ctypes.c_int()
        cnt = (ctypes.c_int64 * 4)()
        _check(_load().pa_alloc_export_host_state(self._h, fo, ctypes.byref(nf), cnt))
        return list(fo[:nf.value]), int(cnt[1]), int(cnt[2]), int(cnt[3])

    def export_state(self):
        """(free list front to back, reference counts)."""
        fo = (ctypes.c_int32 * self.num_blocks)()
        rc = (ctypes.c_int32 * self.num_blocks)()
        nf = ctypes.c_int()
        _check(_load().pa_alloc_export_state(self._h, fo, ctypes.byref(nf), rc))
        return list(fo[:nf.value]), list(rc)
