"""The five decode workloads, drawn from seeded PCG64 streams.

Shapes follow the workloads the PagedAttention pages picture: fixed-size KV
blocks of 16 tokens ("Phase 7 · Document 04 — PagedAttention", §2 Core
Concept, layout sketch), a shared pool of physical blocks handed out in an
arbitrary order (lux-666 notes "PagedAttention", section 最小模型 / minimal
model), and prefixes shared across sequences (same document, §2 "block
sharing" and §3 Mental Model). Sizes, heads and length mixes are the five
synthetic decode batches this library is measured on.

Nothing here computes a block table, a slot or an attention value.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

CONFIG_NAMES = (
    "tiny_mha_d64",          # 4 seqs {5,16,17,40}, 4 heads, D=64, BS=16, 32 blocks
    "gqa4_u128_2048",        # 64 seqs U[128,2048], 32q/8kv, D=128, BS=16
    "mha32_lognormal800",    # 256 seqs lognormal(800, 0.8), MHA 32, D=128, churned pool
    "shared_prefix_cow",     # 128 seqs sharing a 2040-token prefix, 32q/8kv
    "long32k_gqa8",          # 16 seqs x 32768, 64q/8kv, BS in {8,16,32}
)

_CHUNK = 1 << 24  # draws per chunk when filling large pools


def _fill(rng: np.random.Generator, shape, dist: str) -> np.ndarray:
    """fp16 array of `shape` filled in row-major order from `rng`.

    dist "normal": N(0,1); dist "uniform": U(-1,1). Drawn in float32 chunks so
    multi-GB pools do not need a float64 temporary of the same size.
    """
    out = np.empty(int(np.prod(shape)), dtype=np.float16)
    n = out.size
    pos = 0
    while pos < n:
        m = min(_CHUNK, n - pos)
        if dist == "normal":
            vals = rng.standard_normal(m, dtype=np.float32)
        elif dist == "uniform":
            vals = rng.random(m, dtype=np.float32) * np.float32(2.0) - np.float32(1.0)
        else:
            raise ValueError(dist)
        out[pos:pos + m] = vals.astype(np.float16)
        pos += m
    return out.reshape(shape)


def _ceil_div(a: int, b: int) -> int:
    return -(-int(a) // int(b))


@dataclass
class ChurnOp:
    """One allocator operation applied before sequences are placed.

    kind "alloc": a temporary owner `owner` takes `nblocks` blocks.
    kind "free": owner `owner` returns all its blocks.
    """
    kind: str
    owner: int
    nblocks: int = 0


@dataclass
class DecodeBatch:
    """One decode step's inputs: cache contents before the step, plus the new token.

    prefill_lens[i]  tokens of sequence i already in the cache (before the append)
    free_order       initial free-list order of the pool's physical block ids
    churn            allocator traffic to replay before placing the sequences
    q                [S][Hq][D] fp16, the step's queries
    k_pool, v_pool   [NB][BS][Hkv][D] fp16, the shared pools
    k_new, v_new     [S][Hkv][D] fp16, the step's new K/V token per sequence
    scale            fp32 softmax scale (1/sqrt(D) rounded to fp32)
    """
    name: str
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    prefill_lens: np.ndarray
    free_order: np.ndarray
    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    scale: np.float32
    churn: List[ChurnOp] = field(default_factory=list)
    seed: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.prefill_lens.shape[0])

    @property
    def attended_lens(self) -> np.ndarray:
        """Lengths attended in the step: the prefill plus the appended token."""
        return self.prefill_lens + 1


def _scale(head_dim: int) -> np.float32:
    return np.float32(1.0 / math.sqrt(head_dim))


def make_batch(
    name: str,
    rng: np.random.Generator,
    prefill_lens: Sequence[int],
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int,
    num_blocks: int,
    kv_dist: str = "normal",
    shuffle_pool: bool = True,
    churn_fn=None,
    seed: int = 0,
) -> DecodeBatch:
    """Draw a batch in the fixed order: free order, [churn], q, pools, new K/V.

    `prefill_lens` must already have been drawn from `rng` by the caller (it is
    the first draw). `churn_fn(rng)` draws the churn ops, if any.
    """
    lens = np.asarray(prefill_lens, dtype=np.int64)
    if shuffle_pool:
        free_order = rng.permutation(num_blocks).astype(np.int32)
    else:
        free_order = np.arange(num_blocks, dtype=np.int32)
    churn = churn_fn(rng) if churn_fn is not None else []
    S = lens.shape[0]
    q = _fill(rng, (S, num_q_heads, head_dim), "normal")
    k_pool = _fill(rng, (num_blocks, block_size, num_kv_heads, head_dim), kv_dist)
    v_pool = _fill(rng, (num_blocks, block_size, num_kv_heads, head_dim), kv_dist)
    k_new = _fill(rng, (S, num_kv_heads, head_dim), kv_dist)
    v_new = _fill(rng, (S, num_kv_heads, head_dim), kv_dist)
    return DecodeBatch(
        name=name, block_size=block_size, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, num_blocks=num_blocks,
        prefill_lens=lens, free_order=free_order, q=q, k_pool=k_pool,
        v_pool=v_pool, k_new=k_new, v_new=v_new, scale=_scale(head_dim),
        churn=churn, seed=seed,
    )


def _pool_for(attended: np.ndarray, block_size: int, factor: float = 1.25) -> int:
    """Pool size rule of the workloads: `factor` x the blocks the batch needs."""
    need = sum(_ceil_div(int(L), block_size) for L in attended)
    return int(math.ceil(factor * need))


def config1_tiny(seed: int = 1) -> DecodeBatch:
    """4 sequences {5,16,17,40}, 4 heads MHA, D=64, BS=16, 32 permuted blocks,
    K/V U(-1,1), q N(0,1), scale 1/sqrt(64)."""
    rng = np.random.default_rng(seed)
    lens = np.array([5, 16, 17, 40], dtype=np.int64)
    return make_batch("tiny_mha_d64", rng, lens, 4, 4, 64, 16, 32,
                      kv_dist="uniform", seed=seed)


def config2_gqa_batch(seed: int = 2, num_seqs: int = 64, lo: int = 128,
                      hi: int = 2048, num_q_heads: int = 32,
                      num_kv_heads: int = 8, head_dim: int = 128,
                      block_size: int = 16) -> DecodeBatch:
    """64 sequences, lengths U[128,2048], 32 q / 8 kv heads, D=128, BS=16,
    pool 1.25x the blocks needed, shuffled ids. Smaller sizes for quick cases."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi, size=num_seqs, endpoint=True).astype(np.int64)
    nb = _pool_for(lens + 1, block_size)
    return make_batch("gqa4_u128_2048", rng, lens, num_q_heads, num_kv_heads,
                      head_dim, block_size, nb, seed=seed)


def _lognormal_lengths(rng, n, median, sigma, lo, hi):
    x = np.exp(rng.normal(math.log(median), sigma, size=n))
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def config3_mha_lognormal(seed: int = 3, num_seqs: int = 256,
                          median: float = 800.0, sigma: float = 0.8,
                          lo: int = 16, hi: int = 8192, num_heads: int = 32,
                          head_dim: int = 128, block_size: int = 16,
                          churn_ops: int = 10_000,
                          churn_max_blocks: int = 64) -> DecodeBatch:
    """256 sequences with lognormal lengths (median 800, sigma 0.8, clipped to
    [16,8192]), 32 heads MHA, D=128, BS=16, placed after `churn_ops` seeded
    alloc/free operations on the free list."""
    rng = np.random.default_rng(seed)
    lens = _lognormal_lengths(rng, num_seqs, median, sigma, lo, hi)
    nb = _pool_for(lens + 1, block_size)

    def churn(r):
        ops: List[ChurnOp] = []
        live = []          # owners in creation order
        sizes = {}
        free = nb
        for k in range(churn_ops):
            coin = r.random()
            n = int(r.integers(1, churn_max_blocks, endpoint=True))
            u = r.random()
            if coin < 0.5 and free >= n:
                owner = 1_000_000 + k
                ops.append(ChurnOp("alloc", owner, n))
                live.append(owner)
                sizes[owner] = n
                free -= n
            elif live:
                idx = int(u * len(live))
                owner = live.pop(idx)
                ops.append(ChurnOp("free", owner))
                free += sizes.pop(owner)
        # release every survivor, in a seeded order
        for j in r.permutation(len(live)):
            ops.append(ChurnOp("free", live[int(j)]))
        return ops

    return make_batch("mha32_lognormal800", rng, lens, num_heads, num_heads,
                      head_dim, block_size, nb, churn_fn=churn, seed=seed)


@dataclass
class SharedPrefixWorkload:
    """A prefix shared by every sequence, then per-sequence decode steps.

    Sequence 0 holds the prefix; sequences 1..S-1 are forked from it, so every
    prefix block is referenced by all S tables. Sequence i then runs
    `steps[i]` decode steps (append one token, attend) and retires.
    Per-step q / k_new / v_new come from `step_inputs(step, active)`.
    """
    name: str
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    prefix_len: int
    steps: np.ndarray
    free_order: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    scale: np.float32
    seed: int

    @property
    def num_seqs(self) -> int:
        return int(self.steps.shape[0])

    def step_inputs(self, step: int, num_active: int):
        """(q, k_new, v_new) for decode step `step` (0-based) over `num_active`
        sequences, drawn from their own stream keyed by (seed, step)."""
        r = np.random.default_rng([self.seed, 1 + int(step)])
        q = _fill(r, (num_active, self.num_q_heads, self.head_dim), "normal")
        k = _fill(r, (num_active, self.num_kv_heads, self.head_dim), "normal")
        v = _fill(r, (num_active, self.num_kv_heads, self.head_dim), "normal")
        return q, k, v


def config4_shared_prefix(seed: int = 4, num_seqs: int = 128,
                          prefix_len: int = 2040, max_steps: int = 512,
                          num_q_heads: int = 32, num_kv_heads: int = 8,
                          head_dim: int = 128,
                          block_size: int = 16) -> SharedPrefixWorkload:
    """128 sequences sharing a 2040-token prefix (128 blocks, the last holding
    8 tokens), each then running U[1,512] decode steps; 32 q / 8 kv heads."""
    rng = np.random.default_rng(seed)
    steps = rng.integers(1, max_steps, size=num_seqs, endpoint=True).astype(np.int64)
    shared_blocks = _ceil_div(prefix_len, block_size)
    full_shared = prefix_len // block_size
    tail = prefix_len - full_shared * block_size
    private = sum(_ceil_div(tail + int(s), block_size) for s in steps)
    nb = int(math.ceil(1.25 * (shared_blocks + private)))
    free_order = rng.permutation(nb).astype(np.int32)
    k_pool = _fill(rng, (nb, block_size, num_kv_heads, head_dim), "normal")
    v_pool = _fill(rng, (nb, block_size, num_kv_heads, head_dim), "normal")
    return SharedPrefixWorkload(
        name="shared_prefix_cow", block_size=block_size,
        num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        num_blocks=nb, prefix_len=prefix_len, steps=steps,
        free_order=free_order, k_pool=k_pool, v_pool=v_pool,
        scale=_scale(head_dim), seed=seed)


def config5_long_context(block_size: int = 16, seed: int = 5,
                         num_seqs: int = 16, seq_len: int = 32768,
                         num_q_heads: int = 64, num_kv_heads: int = 8,
                         head_dim: int = 128) -> DecodeBatch:
    """16 sequences attending 32768 tokens (32767 in cache + the appended one),
    64 q / 8 kv heads, D=128, one block size from {8,16,32}, permuted pool."""
    rng = np.random.default_rng([seed, block_size])
    lens = np.full(num_seqs, seq_len - 1, dtype=np.int64)
    nb = _pool_for(lens + 1, block_size)
    return make_batch(f"long32k_gqa8_bs{block_size}", rng, lens, num_q_heads,
                      num_kv_heads, head_dim, block_size, nb, seed=seed)


# --- fp8 (E4M3) cache -------------------------------------------------------
@dataclass
class Fp8Cache:
    """An E4M3 KV cache for a batch: byte pools [NB][BS][Hkv][D] and one fp32
    scale per KV head for K and for V."""
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray


def fp8_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Random E4M3 bytes composed from their fields: a fair sign bit, an
    exponent field drawn from 8..14 (magnitudes 2 .. 480, where a per-head
    scaled N(0,1) tensor mostly lands) with more weight on the upper fields, and
    a uniform mantissa. Field 15 with mantissa 7 (NaN) is never drawn."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8)
    exps = np.arange(8, 15)
    w = np.array([1, 1, 2, 3, 4, 4, 3], dtype=np.float64)
    w /= w.sum()
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        m = hi - lo
        sign = rng.integers(0, 2, m, dtype=np.uint8)
        e = rng.choice(exps, m, p=w).astype(np.uint8)
        man = rng.integers(0, 8, m, dtype=np.uint8)
        out[lo:hi] = (sign << 7) | (e << 3) | man
    return out.reshape(shape)


def fp8_finite_codes() -> np.ndarray:
    """The 254 finite E4M3 bytes: every byte but the two NaN codes 0x7F and
    0xFF. They include both zeros, the subnormals (exponent field 0), every
    normal exponent field and the largest magnitudes +-448 (0x7E, 0xFE)."""
    b = np.arange(256, dtype=np.uint8)
    return b[(b & 0x7F) != 0x7F]


def fp8_codes_every_finite(rng: np.random.Generator, shape) -> np.ndarray:
    """E4M3 bytes in which every finite code occurs equally often (the 254
    codes tiled over the array, the last tile cut short) in a seeded random
    order. An array of at least 254 elements holds each finite code at least
    once."""
    n = int(np.prod(shape))
    codes = fp8_finite_codes()
    out = np.resize(codes, n)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        rng.shuffle(out[lo:hi])
    return out.reshape(shape)


def fp8_cache(batch: "DecodeBatch", seed: int = 100, every_code: bool = False) -> Fp8Cache:
    """An E4M3 cache with the shape of `batch`'s pools, from its own stream
    (draw order: k_pool, v_pool, k_scale, v_scale); scales U[0.002, 0.02].
    Codes come from `fp8_codes` (the magnitudes a scaled N(0,1) tensor
    mostly takes), or with `every_code` from `fp8_codes_every_finite` (each
    finite code equally often)."""
    rng = np.random.default_rng(seed)
    shape = batch.k_pool.shape
    hkv = shape[2]
    gen = fp8_codes_every_finite if every_code else fp8_codes
    k = gen(rng, shape)
    v = gen(rng, shape)
    ks = rng.uniform(0.002, 0.02, hkv).astype(np.float32)
    vs = rng.uniform(0.002, 0.02, hkv).astype(np.float32)
    return Fp8Cache(k, v, ks, vs)
