// Shared-prefix decode on the 5th-generation tensor cores: the prefix kernel
// of pa_decode_attention_shared_prefix and its launcher (the attention
// kernel's prefix mode, which folds this kernel's partial records into each
// sequence's result when the suffixes are long, lives with the attention
// kernel).
#include "pa_device.cuh"
#include "pa_tma.h"

#include <mutex>

namespace {

// ------------------------------------------------------ shared prefix ---
// Sequences that begin with the same physical blocks (a shared prompt prefix:
// "Phase 7 · Document 04 — PagedAttention", §2 block sharing and §3 Mental
// Model; lux-666 notes "PagedAttention", prefix sharing) attend those blocks
// with the same K and V rows, so for one KV head the prefix is a dense
// contraction: S = Q K^T with Q the query rows of every sharing sequence
// (rows (sequence, query head of the group), 128 per CTA) and K the prefix's
// tokens, then O = P V. The prefix kernel runs it on the 5th-generation
// tensor cores: Q, K and V sit in shared memory as 128-byte-swizzled operand
// tiles, S and O accumulate in tensor memory (TMEM) and P is written over
// its S in TMEM, whence the PV MMA reads it; one thread issues each kind of
// MMA, a warp each streams the K and V tiles with TMA, and four warps (one
// TMEM lane quarter each, one query row per thread) run the softmax. The
// prefix's tokens are split into chunks across CTAs and each chunk into
// sub-chunks of up to 128 tokens; a row's online softmax runs over its
// chunk's sub-chunks, and each (chunk, sequence, KV head) leaves one partial
// record (the layout the merges use). The attention kernel then streams each
// sequence's remaining blocks and merges the prefix chunks' records into that
// sequence's result.
constexpr int kPfxRows = 128;                   // query rows per CTA = TMEM lanes
constexpr int kPfxTok = 128;                    // tokens per sub-chunk (MMA N of S)
constexpr int kPfxSoftmaxWarps = 4;             // warps 0-3: one TMEM lane quarter each
constexpr int kPfxWarpK = 4;                    // TMA of K tiles
constexpr int kPfxWarpS = 5;                    // S = Q K^T issuer; owns the TMEM allocation
constexpr int kPfxWarpPV = 6;                   // O = P V issuer
constexpr int kPfxWarpV = 7;                    // TMA of V tiles
constexpr int kPfxThreads = 8 * 32;
constexpr int kPfxKStages = 3;                  // K tiles in flight (S runs ahead)
constexpr int kPfxVStages = 3;                  // V tiles in flight
constexpr int kMaxPfxChunks = 32;
constexpr int kPfxTmemCols = 512;               // S[2] (P over S) and O[2], 128 columns each
constexpr int kPfxTile = kPfxTok * 256;         // one operand tile: 128 rows x 128 fp16
// barriers, then the 1024-aligned tiles Q, K[stages], V[stages]
constexpr int kPfxHead = 256;
constexpr int kPfxSmem = 1024 + kPfxHead + (1 + kPfxKStages + kPfxVStages) * kPfxTile;
constexpr int kFusedSuffixTokens = 32;          // fused mode: the longest suffix past the prefix
constexpr int kMaxCluster = 8;                  // fused mode: prefix chunks (cluster size) at most

struct PrefixParams {
  const __half* q;
  const int32_t* prefix_blocks;  // [num_prefix_blocks] physical ids shared by every sequence
  float* records;                // prefix records [nchunks][S][Hkv][rec_floats(G, D)]
  int32_t* err;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int prefix_blocks_n;
  int chunk_blocks;              // prefix blocks per chunk
  float qscale;                  // scale * log2(e)
  // fused mode (every suffix at most kFusedSuffixTokens tokens): the chunks
  // of one (row tile, KV head) form a cluster, merge their partials through
  // distributed shared memory and attend each sequence's suffix themselves
  const int32_t* block_table;    // [S][max_blocks]
  const int32_t* seq_lens;       // [S]
  const __half* k_pool;          // the pools, read row by row for the suffix
  const __half* v_pool;
  long long block_stride;        // values from one pool block to the next
  __half* out;                   // [S][Hq][D]
  int max_blocks;
};

// Shared-memory helpers of a thread-block cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// The same shared-memory address in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// ---- tcgen05 ----------------------------------------------------------------
// Shared-memory operand descriptor: a tile of rows of 128 bytes with the
// 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)), 8-row
// groups `sbo` bytes apart; `lbo` is the distance between the two 64-value
// halves of an MN-major operand (unused for K-major tiles).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of an M=128 x N MMA, fp16 A and B, fp32 accumulate;
// A K-major, B K-major or (b_mn) MN-major.
__device__ __forceinline__ uint32_t f16_idesc(int n, bool b_mn) {
  return (1u << 4) | (b_mn ? 1u << 16 : 0u) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// The same MMA with A read from tensor memory: row i of A in lane i, two
// fp16 values per 32-bit column (the lower K index in the low half).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 16 / 32 consecutive fp32 columns of this thread's TMEM lane; returns after
// the load has completed.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n\ttcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 / 8 consecutive 32-bit columns of this thread's TMEM lane; returns after
// the store has completed.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};\n\ttcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Fused mode: the rows one CTA of a cluster of C finishes, [c * 128 / C,
// (c + 1) * 128 / C) of the row tile, and the sequences they belong to.
// Their suffix rows (the tokens past the prefix, at most kFusedSuffixTokens
// per sequence) are asked of L2 early, so the end of the kernel finds them
// there; called by the four softmax warps while they wait for the first S.
template <int BS, int G>
__device__ __forceinline__ void prefetch_suffix_rows(const PrefixParams& p, int kvh, int c) {
  constexpr int D = 128;
  const int C = gridDim.z, rpc = kPfxRows / C;
  const int r0 = blockIdx.x * kPfxRows + c * rpc;
  const int s_lo = r0 / G, s_hi = min(p.num_seqs, (r0 + rpc + G - 1) / G);
  const int P = p.prefix_blocks_n;
  const int ntok = (p.max_blocks - P) * BS;
  for (int i = threadIdx.x; i < (s_hi - s_lo) * ntok; i += kPfxSoftmaxWarps * 32) {
    const int sq = s_lo + i / ntok, t = i % ntok;
    const int L = min(p.seq_lens[sq], p.max_blocks * BS);
    if (t >= L - P * BS) continue;
    const int blk = p.block_table[static_cast<long long>(sq) * p.max_blocks + P + t / BS];
    if (blk < 0 || blk >= p.num_blocks) continue;
    const long long off = static_cast<long long>(blk) * p.block_stride +
                          (static_cast<long long>(t % BS) * p.num_kv_heads + kvh) * D;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.k_pool + off));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.k_pool + off + 64));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.v_pool + off));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.v_pool + off + 64));
  }
}

// Bulk copy of `bytes` from this CTA's shared memory to shared memory of
// another CTA of the cluster (`dst`, `bar`: shared::cluster addresses there),
// counted on that CTA's barrier.
__device__ __forceinline__ void bulk_copy_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes,
                                                    uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Fused mode, after the cluster barrier: each CTA finishes rows [c * 128 / C,
// (c + 1) * 128 / C) of the tile. Every chunk's CTA staged its rows'
// partials (max and sum in log2 units, then the accumulator; rows of D + 4
// floats) in its own shared memory at `stage`; each now sends the other
// CTAs their rows with one bulk copy each into their `recv` area (slot =
// sender's rank), counted on their `recv_bar`. A row's C partials are merged
// with the log-sum-exp rule, then the row attends its sequence's suffix (the
// tokens past the prefix, at most kFusedSuffixTokens) on CUDA cores,
// continuing that running softmax eight tokens at a time, and the result is
// written as fp16. Eight threads share a row, 16 dimensions each; a score is
// their dot products summed by shuffles within the group.
template <int BS, int G>
__device__ __forceinline__ void fused_merge_and_suffix(const PrefixParams& p, const float* stage,
                                                       float* recv, uint64_t* recv_bar, int kvh,
                                                       int c) {
  constexpr int D = 128, kPad = D + 4, TPR = 8, DPT = D / TPR, kGrp = 8;
  const int C = gridDim.z, rpc = kPfxRows / C;
  const int S = p.num_seqs, P = p.prefix_blocks_n, cap = p.max_blocks * BS;
  const int part = threadIdx.x % TPR;
  const uint32_t rows_bytes = static_cast<uint32_t>(rpc * kPad * 4);
  // ---- exchange: my rows of every other chunk's partials arrive here ----
  if (C > 1) {
    if (threadIdx.x == 0) {
      for (int k = 0; k < C; ++k) {
        if (k == c) continue;
        bulk_copy_s2cluster(cluster_map(smem_addr(recv) + c * rows_bytes, k),
                            smem_addr(stage) + k * rows_bytes, rows_bytes,
                            cluster_map(smem_addr(recv_bar), k));
      }
    }
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(smem_addr(recv_bar), 0) && global_ns() - t0 < kWaitLimitNs) {
    }
  }
  // every lane of a warp runs the same rows loop (rpc is a multiple of 4)
#pragma unroll 1
  for (int lr = threadIdx.x / TPR; lr < rpc; lr += kPfxThreads / TPR) {
    const int rt = c * rpc + lr;
    const int row = blockIdx.x * kPfxRows + rt;
    const int seq = row / G, gg = row % G;
    const bool live = seq < S;
    // this row's suffix length and, meanwhile, its q slice
    int suf = 0;
    uint4 qa = make_uint4(0, 0, 0, 0), qb = qa;
    if (live) {
      const __half* qrow =
          p.q + (static_cast<long long>(seq) * p.num_q_heads + kvh * G + gg) * D + part * DPT;
      qa = *reinterpret_cast<const uint4*>(qrow);
      qb = *reinterpret_cast<const uint4*>(qrow + 8);
      int Ls = p.seq_lens[seq];
      if (Ls < P * BS || Ls > cap) {
        if (part == 0 && gg == 0) atomicOr(p.err, PA_DEVERR_BAD_LEN);
        Ls = Ls < 0 ? 0 : (Ls > cap ? cap : Ls);
      }
      suf = min(max(Ls - P * BS, 0), kFusedSuffixTokens);
    }
    // ---- merge the C chunk partials of the row (local shared memory) ----
    auto src = [&](int k) -> const float* {
      return k == c ? stage + rt * kPad : recv + k * rpc * kPad + lr * kPad;
    };
    float M = -INFINITY;
#pragma unroll 1
    for (int k = 0; k < C; ++k) M = fmaxf(M, src(k)[D]);
    const float mu = M == -INFINITY ? 0.f : M;
    float acc[DPT], L = 0.f;
#pragma unroll
    for (int i = 0; i < DPT; ++i) acc[i] = 0.f;
#pragma unroll 1
    for (int k = 0; k < C; ++k) {
      const float* r = src(k);
      const float mk = r[D];
      if (mk != -INFINITY) {
        const float w = fast_exp2(mk - mu);
        L += w * r[D + 1];
#pragma unroll
        for (int i = 0; i < DPT; i += 4) {
          const float4 v = *reinterpret_cast<const float4*>(r + part * DPT + i);
          acc[i] += w * v.x;
          acc[i + 1] += w * v.y;
          acc[i + 2] += w * v.z;
          acc[i + 3] += w * v.w;
        }
      }
    }
    // ---- the suffix: tokens P * BS .. L - 1 of the sequence ----
    float qv[DPT];
    {
      const __half2* h = reinterpret_cast<const __half2*>(&qa);
      const __half2* h2 = reinterpret_cast<const __half2*>(&qb);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]), f2 = __half22float2(h2[i]);
        qv[2 * i] = f.x;
        qv[2 * i + 1] = f.y;
        qv[8 + 2 * i] = f2.x;
        qv[8 + 2 * i + 1] = f2.y;
      }
    }
    // the suffix's block ids, loaded and checked once
    constexpr int kSufBlocks = (kFusedSuffixTokens + BS - 1) / BS;
    int blk[kSufBlocks];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kSufBlocks; ++j) {
      blk[j] = -1;
      if (j * BS < suf) {
        blk[j] = p.block_table[static_cast<long long>(seq) * p.max_blocks + P + j];
        if (blk[j] < 0 || blk[j] >= p.num_blocks) {
          bad = true;
          blk[j] = -1;
        }
      }
    }
    if (bad && part == 0) atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
    // pool offset of suffix token t of this row's KV head (-1: not read)
    auto row_off = [&](int t) -> long long {
      int b = blk[0];
#pragma unroll
      for (int j = 1; j < kSufBlocks; ++j)
        if (t >= j * BS) b = blk[j];
      if (t >= suf || b < 0) return -1;
      return static_cast<long long>(b) * p.block_stride +
             (static_cast<long long>(t % BS) * p.num_kv_heads + kvh) * D + part * DPT;
    };
    int suf_w = suf;  // the warp's longest suffix: every lane runs the shuffles
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) suf_w = max(suf_w, __shfl_xor_sync(0xffffffffu, suf_w, off));
    // running softmax over the suffix from the merged prefix, eight tokens
    // at a time: all their rows are loaded before any is used
    float m_run = M;
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 1
    for (int t0 = 0; t0 < suf_w; t0 += kGrp) {
      uint4 kx[kGrp][2], vx[kGrp][2];
      bool ok[kGrp];
#pragma unroll
      for (int u = 0; u < kGrp; ++u) {
        const long long off = row_off(t0 + u);
        ok[u] = off >= 0;
        kx[u][0] = ok[u] ? *reinterpret_cast<const uint4*>(p.k_pool + off) : z;
        kx[u][1] = ok[u] ? *reinterpret_cast<const uint4*>(p.k_pool + off + 8) : z;
        vx[u][0] = ok[u] ? *reinterpret_cast<const uint4*>(p.v_pool + off) : z;
        vx[u][1] = ok[u] ? *reinterpret_cast<const uint4*>(p.v_pool + off + 8) : z;
      }
      float sc[kGrp];
#pragma unroll
      for (int u = 0; u < kGrp; ++u) {
        const __half2* h = reinterpret_cast<const __half2*>(&kx[u][0]);
        const __half2* h2 = reinterpret_cast<const __half2*>(&kx[u][1]);
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(h[i]), f2 = __half22float2(h2[i]);
          d = fmaf(qv[2 * i], f.x, d);
          d = fmaf(qv[2 * i + 1], f.y, d);
          d = fmaf(qv[8 + 2 * i], f2.x, d);
          d = fmaf(qv[8 + 2 * i + 1], f2.y, d);
        }
        sc[u] = d;
      }
      float gm = m_run;
#pragma unroll
      for (int u = 0; u < kGrp; ++u) {
        float d = sc[u];
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        sc[u] = ok[u] ? d * p.qscale : -INFINITY;
        gm = fmaxf(gm, sc[u]);
      }
      if (gm != -INFINITY) {
        const float cf = m_run == -INFINITY ? 0.f : fast_exp2(m_run - gm);
        L *= cf;
#pragma unroll
        for (int i = 0; i < DPT; ++i) acc[i] *= cf;
#pragma unroll
        for (int u = 0; u < kGrp; ++u) {
          if (ok[u]) {
            const float w = fast_exp2(sc[u] - gm);
            L += w;
            const __half2* h = reinterpret_cast<const __half2*>(&vx[u][0]);
            const __half2* h2 = reinterpret_cast<const __half2*>(&vx[u][1]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __half22float2(h[i]), f2 = __half22float2(h2[i]);
              acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
              acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
              acc[8 + 2 * i] = fmaf(w, f2.x, acc[8 + 2 * i]);
              acc[8 + 2 * i + 1] = fmaf(w, f2.y, acc[8 + 2 * i + 1]);
            }
          }
        }
        m_run = gm;
      }
    }
    if (live) {
      // the merged prefix and the suffix are relative to m_run (or to the
      // prefix's max when the suffix is empty): the sum L normalises both
      const float inv = L > 0.f ? 1.f / L : 0.f;
      uint4 o0, o1;
      uint32_t* w0 = reinterpret_cast<uint32_t*>(&o0);
      uint32_t* w1 = reinterpret_cast<uint32_t*>(&o1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w0[i] = pack_half2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
        w1[i] = pack_half2(acc[8 + 2 * i] * inv, acc[8 + 2 * i + 1] * inv);
      }
      __half* orow = p.out + (static_cast<long long>(seq) * p.num_q_heads + kvh * G + gg) * D +
                     part * DPT;
      *reinterpret_cast<uint4*>(orow) = o0;
      *reinterpret_cast<uint4*>(orow + 8) = o1;
    }
  }
}

template <int BS, int G, bool FUSED>
__global__ void __launch_bounds__(kPfxThreads, 1)
    paged_prefix_kernel(const PrefixParams p, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  constexpr int D = 128;
  constexpr int HALF = kPfxTile / 2;           // one 64-value half: 128 rows x 128 B
  constexpr int RS = rec_floats(G, D);
  static_assert(kPfxTok % BS == 0 && BS % 16 == 0, "sub-chunks are whole blocks of 16-token boxes");
  extern __shared__ __align__(1024) unsigned char psm[];
  // barriers and flags, then 1024-aligned tiles: Q, K[NK], V[NV]
  constexpr int NK = kPfxKStages, NV = kPfxVStages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(psm);
  uint64_t* k_full = bars;                     // [NK] TMA -> S issuer
  uint64_t* k_empty = bars + NK;               // [NK] S MMAs done with a K tile
  uint64_t* v_full = bars + 2 * NK;            // [NV] TMA -> PV issuer
  uint64_t* v_empty = bars + 2 * NK + NV;      // [NV] PV MMAs done with a V tile
  uint64_t* s_full = bars + 2 * NK + 2 * NV;   // [2] S buffer written
  uint64_t* s_free = s_full + 2;               // [2] PV MMAs done with the P written over S
  uint64_t* p_full = s_full + 4;               // [2] P written (4 softmax warps)
  uint64_t* o_full = s_full + 6;               // [2] O buffer written
  uint64_t* o_free = s_full + 8;               // [2] O buffer read (4 softmax warps)
  uint64_t* mma_done = s_full + 10;            // [2] every MMA of an issuer completed
  constexpr int kBars = 2 * NK + 2 * NV + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* recv_bar = bars + kBars + 1;       // fused mode: the other chunks' partials arrived
  static_assert(kBars * 8 + 16 <= 256, "barriers fit below the tiles");
  const uint32_t sbase = smem_addr(psm);
  unsigned char* tiles = psm + (((sbase + kPfxHead + 1023u) & ~1023u) - sbase);
  unsigned char* q_s = tiles;
  unsigned char* k_s = tiles + kPfxTile;                       // [NK]
  unsigned char* v_s = tiles + (1 + NK) * kPfxTile;            // [NV]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y, c = blockIdx.z;
  const int S = p.num_seqs;
  const int tok_lo = c * p.chunk_blocks * BS;
  const int tok_hi = max(tok_lo, min(p.prefix_blocks_n, (c + 1) * p.chunk_blocks) * BS);
  const int nsub = (tok_hi - tok_lo + kPfxTok - 1) / kPfxTok;
  auto sub_len = [&](int t) { return min(kPfxTok, tok_hi - (tok_lo + t * kPfxTok)); };

  if (threadIdx.x == 0) {
    // p_full and o_free count the four softmax warps; the others one arrival
    // (a TMA transaction count or an MMA commit)
    for (int i = 0; i < kBars; ++i) {
      const uint64_t* b = &bars[i];
      const bool softmax = (b >= p_full && b < p_full + 2) || (b >= o_free && b < o_free + 2);
      mbar_init(smem_addr(&bars[i]), softmax ? kPfxSoftmaxWarps : 1);
    }
    *abort_flag = 0;
    if (FUSED) {
      // the other C - 1 chunks of the cluster each send this CTA's rows of
      // their partials (see the end of the kernel)
      const uint32_t rb = smem_addr(recv_bar);
      mbar_init(rb, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      mbar_arrive_expect_tx(rb, (gridDim.z - 1) * (kPfxRows / gridDim.z) * (128 + 4) * 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Everything launched before this kernel has completed: the attention
  // kernel that follows may start streaming (it waits for this kernel only
  // before it reads the prefix records).
  asm volatile("griddepcontrol.launch_dependents;");
  const bool tma_warp = warp == kPfxWarpK || warp == kPfxWarpV;
  uint32_t tmem = 0;
  if (!tma_warp) {
    // the TMA warps start streaming at once; the other six warps stage Q and
    // allocate TMEM, then meet on a named barrier
    if (warp == kPfxWarpS) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_addr(tmem_slot)),
                   "n"(kPfxTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Q rows -> shared memory as the K-major A operand (zero rows past the
    // batch); every load of a thread is in flight before its first store
    constexpr int kQThreads = kPfxThreads - 64;
    const int qt = warp < kPfxWarpK ? threadIdx.x : threadIdx.x - 32;  // 0..191
    constexpr int kPer = (kPfxRows * (D / 8) + kQThreads - 1) / kQThreads;
    uint4 v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = qt + i * kQThreads;
      const int r = e / (D / 8), ch = e % (D / 8);
      const int row = blockIdx.x * kPfxRows + r, seq = row / G, gg = row % G;
      v[i] = make_uint4(0, 0, 0, 0);
      if (e < kPfxRows * (D / 8) && seq < S)
        v[i] = __ldg(reinterpret_cast<const uint4*>(
            p.q + (static_cast<long long>(seq) * p.num_q_heads + kvh * G + gg) * D) + ch);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = qt + i * kQThreads;
      const int r = e / (D / 8), ch = e % (D / 8);
      if (e < kPfxRows * (D / 8))
        *reinterpret_cast<uint4*>(q_s + (ch >> 3) * HALF + r * 128 +
                                  (((ch & 7) ^ (r & 7)) << 4)) = v[i];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(kPfxThreads - 64) : "memory");
    tc_fence_after();
    tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  }

  int issued = 0;  // sub-chunks whose copies a TMA warp issued
  if (tma_warp) {
    // ---- TMA: the K (or V) tile of each sub-chunk, 16-token boxes per half ----
    const bool is_k = warp == kPfxWarpK;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    const int nst = is_k ? NK : NV;
    unsigned char* ring = is_k ? k_s : v_s;
    // block ids of a sub-chunk: one per lane, all loaded at once; the next
    // sub-chunk's are in flight while this one's copies are issued
    auto load_ids = [&](int t) {
      const int nb = sub_len(t) / BS;
      int id = 0;
      if (lane < nb) {
        id = __ldg(p.prefix_blocks + (tok_lo + t * kPfxTok) / BS + lane);
        if (id < 0 || id >= p.num_blocks) {
          if (is_k) atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
          id = 0;  // an in-range block keeps the byte count; the result is flagged
        }
      }
      return id;
    };
    int next_ids = nsub > 0 ? load_ids(0) : 0;
    for (int t = 0; t < nsub; ++t, ++issued) {
      const int st = t % nst, n = sub_len(t);
      const int ids = next_ids;
      if (t >= nst &&
          !warp_wait_phase(smem_addr(&empty[st]), ((t / nst) - 1) & 1, abort_flag, p.err))
        break;
      const uint32_t dst = smem_addr(ring + st * kPfxTile), bar = smem_addr(&full[st]);
      if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * 256u);
      for (int j = 0; j < n / BS; ++j) {
        const int phys = __shfl_sync(0xffffffffu, ids, j);
        if (lane == 0) {
#pragma unroll
          for (int sb = 0; sb < BS / 16; ++sb) {
            const uint32_t off = static_cast<uint32_t>(j * BS + sb * 16) * 128u;
            tma_load_4d(dst + off, map, 0, sb * 16, kvh, phys, bar);
            tma_load_4d(dst + HALF + off, map, 64, sb * 16, kvh, phys, bar);
          }
        }
      }
      if (t + 1 < nsub) next_ids = load_ids(t + 1);
      __syncwarp();
    }
    if (*abort_flag) {
      // the last copies issued into each stage land before the CTA exits
      for (int t = issued > nst ? issued - nst : 0; t < issued; ++t) {
        const unsigned long long w0 = global_ns();
        while (!mbar_try_wait(smem_addr(&full[t % nst]), (t / nst) & 1) &&
               global_ns() - w0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == kPfxWarpS) {
    // ---- S issuer: S_t = Q K_t^T into TMEM buffer t % 2 ----
    const uint32_t qa = smem_addr(q_s);
    for (int t = 0; t < nsub; ++t) {
      const int st = t % NK, b = t & 1;
      if (!warp_wait_phase(smem_addr(&k_full[st]), (t / NK) & 1, abort_flag, p.err)) break;
      if (t >= 2 && !warp_wait_phase(smem_addr(&s_free[b]), ((t - 2) >> 1) & 1, abort_flag, p.err))
        break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t kb = smem_addr(k_s + st * kPfxTile);
        const uint32_t id = f16_idesc(sub_len(t), false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * HALF + (k & 3) * 32;
          tc_mma(tmem + b * kPfxTok, sw128_desc(qa + off, 16, 1024),
                 sw128_desc(kb + off, 16, 1024), id, k > 0);
        }
        tc_commit(smem_addr(&s_full[b]));
        tc_commit(smem_addr(&k_empty[st]));
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(smem_addr(&mma_done[0]));
    __syncwarp();
    const unsigned long long w0 = global_ns();
    while (!mbar_try_wait(smem_addr(&mma_done[0]), 0) && global_ns() - w0 < kWaitLimitNs) {
    }
  } else if (warp == kPfxWarpPV) {
    // ---- PV issuer: O_t = P_t V_t into TMEM buffer 2 + t % 2 ----
    for (int t = 0; t < nsub; ++t) {
      const int st = t % NV, b = t & 1;
      if (!warp_wait_phase(smem_addr(&p_full[b]), (t >> 1) & 1, abort_flag, p.err)) break;
      if (!warp_wait_phase(smem_addr(&v_full[st]), (t / NV) & 1, abort_flag, p.err)) break;
      if (t >= 2 && !warp_wait_phase(smem_addr(&o_free[b]), ((t - 2) >> 1) & 1, abort_flag, p.err))
        break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t vb = smem_addr(v_s + st * kPfxTile);
        const uint32_t id = f16_idesc(D, true);
        const int n = sub_len(t);
        // A = P over S buffer b: 16 tokens per MMA, 8 TMEM columns
        for (int k = 0; k < n / 16; ++k)
          tc_mma_ts(tmem + (2 + b) * kPfxTok, tmem + b * kPfxTok + 8 * k,
                    sw128_desc(vb + k * 2048, HALF, 1024), id, k > 0);
        tc_commit(smem_addr(&o_full[b]));
        tc_commit(smem_addr(&v_empty[st]));
        tc_commit(smem_addr(&s_free[b]));
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(smem_addr(&mma_done[1]));
    __syncwarp();
    const unsigned long long w0 = global_ns();
    while (!mbar_try_wait(smem_addr(&mma_done[1]), 0) && global_ns() - w0 < kWaitLimitNs) {
    }
  } else {
    // ---- softmax warps: query row r = 32 * warp + lane (TMEM lane r) ----
    if constexpr (FUSED) prefetch_suffix_rows<BS, G>(p, kvh, c);
    const int r = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float o[D];
#pragma unroll
    for (int i = 0; i < D; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f, alpha_prev = 0.f;
    bool ok = true;
    // fold O_t (relative to the max after sub-chunk t) into o
    auto fold = [&](int t, float alpha) -> bool {
      const int b = t & 1;
      if (!warp_wait_phase(smem_addr(&o_full[b]), (t >> 1) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        tmem_ld32(lane_base + (2 + b) * kPfxTok + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c0 + i] = fmaf(o[c0 + i], alpha, v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&o_free[b]));
      return true;
    };
    for (int t = 0; t < nsub && ok; ++t) {
      const int n = sub_len(t), b = t & 1;
      if (!warp_wait_phase(smem_addr(&s_full[b]), (t >> 1) & 1, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t sa = lane_base + b * kPfxTok;
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      int c0 = 0;
      for (; c0 + 32 <= n; c0 += 32) {
        float v[32];
        tmem_ld32(sa + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], v[i] * p.qscale);
      }
      if (c0 < n) {
        float v[16];
        tmem_ld16(sa + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], v[i] * p.qscale);
      }
      const float mn = fmaxf(m, fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])));
      const float alpha = fast_exp2(m - mn);
      m = mn;
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
      // P = exp2(S * qscale - m) as fp16 pairs, written over the S columns
      // already read: tokens c0 .. c0+2k-1 go to columns c0/2 .. c0/2+k-1
      auto emit = [&](const float* v, uint32_t* h, int cnt) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < cnt) {
            const float e0 = fast_exp2(fmaf(v[2 * i], p.qscale, -mn));
            const float e1 = fast_exp2(fmaf(v[2 * i + 1], p.qscale, -mn));
            sum4[(2 * i) & 3] += e0;
            sum4[(2 * i + 1) & 3] += e1;
            h[i] = pack_half2(e0, e1);
          }
        }
      };
      for (c0 = 0; c0 + 32 <= n; c0 += 32) {
        float v[32];
        tmem_ld32(sa + c0, v);
        uint32_t h[16];
        emit(v, h, 16);
        tmem_st16(sa + c0 / 2, h);
      }
      if (c0 < n) {
        float v[16];
        tmem_ld16(sa + c0, v);
        uint32_t h[16];
        emit(v, h, 8);
        tmem_st8(sa + c0 / 2, h);
      }
      l = l * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&p_full[b]));
      // O of the previous sub-chunk, folded while the tensor cores run this one's
      if (t > 0) ok = fold(t - 1, alpha_prev);
      alpha_prev = alpha;
    }
    if (ok && nsub > 0) ok = fold(nsub - 1, alpha_prev);
    // ---- the chunk's partial records of this warp's 32 rows ----
    // Every MMA has completed (the last O was folded), so the K tiles are
    // free: each warp stages its rows there (16.5 KB, rows padded to 132
    // floats against bank conflicts) and writes each sequence's G rows as one
    // contiguous run, 512 bytes per store instruction.
    constexpr int kPad = D + 4;
    float* stage = reinterpret_cast<float*>(k_s) + warp * 32 * kPad;
#pragma unroll
    for (int i = 0; i < D; i += 4)
      *reinterpret_cast<float4*>(stage + lane * kPad + i) =
          make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
    if constexpr (FUSED) {
      // the cluster merges the rows from here (see the end of the kernel);
      // bulk copies read them, so the writes are ordered for that proxy
      stage[lane * kPad + D] = m;
      stage[lane * kPad + D + 1] = l;
      fence_proxy_async_smem();
    }
    __syncwarp();
    const int row = blockIdx.x * kPfxRows + r, seq = row / G, gg = row % G;
    const bool write = !FUSED && ok && !*abort_flag;
    if (seq < S && write) {
      float* rec = p.records + ((static_cast<long long>(c) * S + seq) * p.num_kv_heads + kvh) * RS;
      rec[G * D + 2 * gg] = m;
      rec[G * D + 2 * gg + 1] = l;
    }
    if (write) {
      // the warp's rows 32w .. 32w+31 belong to sequences row / G; a record's
      // G rows are contiguous ([G][D] floats)
      const int row0 = blockIdx.x * kPfxRows + warp * 32;
      for (int e = lane; e < 32 * (D / 4); e += 32) {
        const int rr = e / (D / 4), i4 = e % (D / 4);
        const int rw = row0 + rr, sq = rw / G, g2 = rw % G;
        if (sq < S) {
          float* rec =
              p.records + ((static_cast<long long>(c) * S + sq) * p.num_kv_heads + kvh) * RS;
          *reinterpret_cast<float4*>(rec + g2 * D + 4 * i4) =
              *reinterpret_cast<const float4*>(stage + rr * kPad + 4 * i4);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kPfxWarpS) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(kPfxTmemCols)
                 : "memory");
  }
  if constexpr (FUSED) {
    // Every CTA of the cluster (the chunks of this row tile and KV head)
    // reaches both barriers, whatever happened before: the first makes all
    // staged partials visible, the second keeps each CTA's shared memory
    // alive until the others have read it.
    cluster_sync_all();
    fused_merge_and_suffix<BS, G>(p, reinterpret_cast<const float*>(k_s),
                                  reinterpret_cast<float*>(v_s), recv_bar, kvh, c);
    cluster_sync_all();
  }
}


// --------------------------------------------------------------- host ---
// --- shared prefix ---------------------------------------------------------
// Prefix chunks: as many (row tiles x KV heads x chunks) CTAs as fit one wave
// of one CTA per SM (at least one chunk), at most kMaxPfxChunks and at most
// one per prefix block.
struct PfxGeom {
  int row_tiles, chunks, chunk_blocks;
};
PfxGeom prefix_geometry(int S, int G, int Hkv, int P, int sm_count) {
  PfxGeom g;
  g.row_tiles = (S * G + kPfxRows - 1) / kPfxRows;
  const long long base = static_cast<long long>(g.row_tiles) * Hkv;
  long long c = sm_count / base;
  if (c > kMaxPfxChunks) c = kMaxPfxChunks;
  if (c > P) c = P;
  if (c < 1) c = 1;
  g.chunk_blocks = static_cast<int>((P + c - 1) / c);
  g.chunks = (P + g.chunk_blocks - 1) / g.chunk_blocks;
  return g;
}

// Fused mode: the chunks of one (row tile, KV head) form a cluster, so their
// count is the cluster size: the largest of 8, 4, 2 (at most one chunk per
// prefix block) whose grid still fits one wave of one CTA per SM, else 1.
PfxGeom fused_prefix_geometry(int S, int G, int Hkv, int P, int sm_count) {
  PfxGeom g;
  g.row_tiles = (S * G + kPfxRows - 1) / kPfxRows;
  const long long base = static_cast<long long>(g.row_tiles) * Hkv;
  int c = kMaxCluster;
  while (c > 1 && (c > P || base * c > sm_count)) c /= 2;
  g.chunks = c;
  g.chunk_blocks = (P + c - 1) / c;
  return g;
}

template <int BS, int G, bool FUSED>
pa_status launch_prefix(const PrefixParams& pp, const PfxGeom& geo, const void* k_pool,
                        const void* v_pool, int Hkv, int NB, long long stride_bytes,
                        const pa::DeviceInfo& dev, cudaStream_t stream) {
  constexpr int D = 128;
  auto kernel = paged_prefix_kernel<BS, G, FUSED>;
  {
    static std::mutex mu;
    static bool set[pa::kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev.device]) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kPfxSmem);
      if (e != cudaSuccess) return pa::cuda_fail(e, "cudaFuncSetAttribute(prefix)");
      set[dev.device] = true;
    }
  }
  CUtensorMap kmap, vmap;
  pa::MapKey kk{dev.device, k_pool, D, BS, Hkv, NB, 1, 16, 2, stride_bytes};
  pa::MapKey vk{dev.device, v_pool, D, BS, Hkv, NB, 1, 16, 2, stride_bytes};
  if (pa_status s = pa::pool_tensor_map(kk, &kmap)) return s;
  if (pa_status s = pa::pool_tensor_map(vk, &vmap)) return s;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(geo.row_tiles), static_cast<unsigned>(Hkv),
                    static_cast<unsigned>(geo.chunks));
  lc.blockDim = dim3(kPfxThreads);
  lc.dynamicSmemBytes = kPfxSmem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (FUSED && geo.chunks > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = static_cast<unsigned>(geo.chunks);
    lc.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&lc, kernel, pp, kmap, vmap);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return pa::cuda_fail(e, "shared-prefix kernel launch");
  pa::count_launch();
  return PA_OK;
}

// Whether clusters of `chunks` prefix CTAs can be resident on this device
// (checked once per device and cluster size).
template <int BS, int G>
bool fused_prefix_fits(const PfxGeom& geo, const pa::DeviceInfo& dev) {
  if (geo.chunks <= 1) return true;
  static std::mutex mu;
  static signed char known[pa::kMaxDevices][kMaxCluster + 1] = {};
  std::lock_guard<std::mutex> lock(mu);
  signed char& k = known[dev.device][geo.chunks];
  if (k == 0) {
    auto kernel = paged_prefix_kernel<BS, G, true>;
    k = -1;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfxSmem) ==
        cudaSuccess) {
      cudaLaunchConfig_t lc = {};
      lc.gridDim = dim3(static_cast<unsigned>(geo.row_tiles), 1, static_cast<unsigned>(geo.chunks));
      lc.blockDim = dim3(kPfxThreads);
      lc.dynamicSmemBytes = kPfxSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = static_cast<unsigned>(geo.chunks);
      lc.attrs = attr;
      lc.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &lc) == cudaSuccess && clusters > 0)
        k = 1;
    }
    cudaGetLastError();  // a refused query is an answer, not an error of the call
  }
  return k > 0;
}

template <int BS, int G>
pa_status prefix_pass(const pa::SharedPrefixCall& call, const pa::DeviceInfo& dev,
                      cudaStream_t s, bool* suffix_pass, int* chunks) {
  PrefixParams pp;
  pp.q = static_cast<const __half*>(call.q);
  pp.prefix_blocks = call.prefix_blocks;
  pp.records = call.records;
  pp.err = call.err;
  pp.num_seqs = call.num_seqs;
  pp.num_q_heads = call.num_q_heads;
  pp.num_kv_heads = call.num_kv_heads;
  pp.num_blocks = call.num_blocks;
  pp.prefix_blocks_n = call.prefix_blocks_n;
  pp.qscale = call.qscale;
  pp.block_table = call.block_table;
  pp.seq_lens = call.seq_lens;
  pp.k_pool = static_cast<const __half*>(call.k_pool);
  pp.v_pool = static_cast<const __half*>(call.v_pool);
  pp.block_stride = call.block_stride_bytes / 2;
  pp.out = static_cast<__half*>(call.out);
  pp.max_blocks = call.max_blocks;
  const int S = call.num_seqs, Hkv = call.num_kv_heads, P = call.prefix_blocks_n;
  // one launch when every suffix is short and the clusters fit
  if ((call.max_blocks - P) * BS <= kFusedSuffixTokens) {
    const PfxGeom fg = fused_prefix_geometry(S, G, Hkv, P, dev.sm_count);
    if (fused_prefix_fits<BS, G>(fg, dev)) {
      pp.chunk_blocks = fg.chunk_blocks;
      *suffix_pass = false;
      *chunks = fg.chunks;
      return launch_prefix<BS, G, true>(pp, fg, call.k_pool, call.v_pool, Hkv, call.num_blocks,
                                        call.block_stride_bytes, dev, s);
    }
  }
  const PfxGeom geo = prefix_geometry(S, G, Hkv, P, dev.sm_count);
  pp.chunk_blocks = geo.chunk_blocks;
  *suffix_pass = true;
  *chunks = geo.chunks;
  return launch_prefix<BS, G, false>(pp, geo, call.k_pool, call.v_pool, Hkv, call.num_blocks,
                                     call.block_stride_bytes, dev, s);
}

}  // namespace

namespace pa {

// The most prefix chunks the unfused mode writes records for.
int max_prefix_chunks() { return kMaxPfxChunks; }

pa_status launch_shared_prefix(const SharedPrefixCall& call, const DeviceInfo& dev,
                               cudaStream_t stream, bool* suffix_pass, int* chunks) {
  const int G = call.num_q_heads / call.num_kv_heads, BS = call.block_size;
#define PA_PFX_CASE(bs, g) \
  if (BS == bs && G == g) return prefix_pass<bs, g>(call, dev, stream, suffix_pass, chunks);
  PA_PFX_CASE(16, 1) PA_PFX_CASE(16, 2) PA_PFX_CASE(16, 4) PA_PFX_CASE(16, 8)
  PA_PFX_CASE(32, 1) PA_PFX_CASE(32, 2) PA_PFX_CASE(32, 4) PA_PFX_CASE(32, 8)
#undef PA_PFX_CASE
  return fail(PA_ERR_UNSUPPORTED, "pa_decode_attention_shared_prefix: unsupported shape");
}

}  // namespace pa
