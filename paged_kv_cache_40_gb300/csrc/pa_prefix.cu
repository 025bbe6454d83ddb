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
// chunk's sub-chunks. O accumulates in TMEM over the whole chunk: the
// softmax takes P against a reference max that moves only when a
// sub-chunk's max exceeds it by more than 2^8, and only then rescales O in
// TMEM (the "online softmax" of the pages with a lazy rescale: the result is
// the same ratio, every exponent stays at most 2^8). Each (chunk, sequence,
// KV head) leaves one partial record (the layout the merges use). The
// attention kernel then streams each sequence's remaining blocks and merges
// the prefix chunks' records into that sequence's result; in the fused mode
// the chunks of a cluster merge their partials themselves.
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
constexpr int kPfxTmemCols = 512;               // S[2] (P over S) at 0 and 128, O at 256
constexpr int kPfxOCol = 256;                   // O accumulates here over every sub-chunk
constexpr float kRescaleLog2 = 8.f;             // the running max moves by more than this only
constexpr int kPfxTile = kPfxTok * 256;         // one operand tile: 128 rows x 128 fp16
// barriers, then the 1024-aligned tiles Q, K[stages], V[stages]
constexpr int kPfxHead = 256;
constexpr int kPfxSmem = 1024 + kPfxHead + (1 + kPfxKStages + kPfxVStages) * kPfxTile;
constexpr int kFusedSuffixTokens = 32;          // fused mode: the longest suffix past the prefix
constexpr int kMaxSuffixSub = 2;                // fused mode: suffix sub-chunks per CTA at most
// fused mode: a row's partial as it crosses the cluster: the accumulator
// divided by its sum as 128 fp16, then max and sum (fp32), padded to 16 bytes
constexpr int kXRow = 128 * 2 + 16;
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
  // of one (row tile, KV head) form a cluster; each attends the suffixes of
  // the rows it finishes as extra sub-chunks, and the cluster merges the
  // partials through distributed shared memory
  const int32_t* block_table;    // [S][max_blocks]
  const int32_t* seq_lens;       // [S]
  __half* out;                   // [S][Hq][D]
  int max_blocks;
};

// Shared-memory helpers of a thread-block cluster. The cluster barrier is
// split: every thread of every CTA arrives, and a wait returns once all have.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
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
// 32 consecutive fp32 columns of this thread's TMEM lane; returns after the
// load has completed.
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

// The 128 fp32 columns of this thread's TMEM lane from `taddr` (an S row)
// in one load; returns after it has completed.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,"
      "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
      "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
        "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
        "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
        "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
        "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
        "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}
// 64 / 32 consecutive 32-bit columns of this thread's lane; returns after the
// store has completed.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&h)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]), "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]),
        "r"(h[8]), "r"(h[9]), "r"(h[10]), "r"(h[11]), "r"(h[12]), "r"(h[13]), "r"(h[14]), "r"(h[15]),
        "r"(h[16]), "r"(h[17]), "r"(h[18]), "r"(h[19]), "r"(h[20]), "r"(h[21]), "r"(h[22]), "r"(h[23]),
        "r"(h[24]), "r"(h[25]), "r"(h[26]), "r"(h[27]), "r"(h[28]), "r"(h[29]), "r"(h[30]), "r"(h[31]),
        "r"(h[32]), "r"(h[33]), "r"(h[34]), "r"(h[35]), "r"(h[36]), "r"(h[37]), "r"(h[38]), "r"(h[39]),
        "r"(h[40]), "r"(h[41]), "r"(h[42]), "r"(h[43]), "r"(h[44]), "r"(h[45]), "r"(h[46]), "r"(h[47]),
        "r"(h[48]), "r"(h[49]), "r"(h[50]), "r"(h[51]), "r"(h[52]), "r"(h[53]), "r"(h[54]), "r"(h[55]),
        "r"(h[56]), "r"(h[57]), "r"(h[58]), "r"(h[59]), "r"(h[60]), "r"(h[61]), "r"(h[62]), "r"(h[63])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
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

// Fused mode: each CTA finishes rows [c * 128 / C, (c + 1) * 128 / C) of the
// tile, whose suffix tokens its own last sub-chunks attended. Every chunk's
// CTA staged each row's partial in its own shared memory (`stage`, rows of
// kXRow bytes: the accumulator divided by the sum as fp16, then max and sum
// in log2 units as fp32) and sent the rows of this CTA's slice with bulk
// copies into `recv` at [sender's rank][row in the slice], counted on
// `recv_bar`. Once the C - 1 other chunks' rows have landed this CTA arrives
// on the cluster barrier that the end of the kernel waits for (so no CTA
// leaves while its staged rows are still being copied out). A row's C
// partials are then merged with the log-sum-exp rule and the result is
// written as fp16, eight threads per row; thread `part` of a row takes the
// dimensions 4 * part + 32 * k .. + 3 (k < 4), so that the row's eight threads
// read 64 contiguous bytes of a partial at a time.
template <int G>
__device__ __forceinline__ void fused_merge(const PrefixParams& p, const unsigned char* stage,
                                            const unsigned char* recv, uint64_t* recv_bar,
                                            int kvh, int c) {
  constexpr int D = 128, TPR = 8;
  const int C = gridDim.z, rpc = kPfxRows / C;
  const int part = threadIdx.x % TPR;
  if (C > 1) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(smem_addr(recv_bar), 0)) {
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicOr(p.err, PA_DEVERR_TIMEOUT);
        break;
      }
    }
  }
  cluster_arrive();
#pragma unroll 1
  for (int lr = threadIdx.x / TPR; lr < rpc; lr += kPfxThreads / TPR) {
    const int rt = c * rpc + lr;
    const int row = blockIdx.x * kPfxRows + rt;
    const int seq = row / G, gg = row % G;
    if (seq >= p.num_seqs) continue;
    auto src = [&](int k) -> const unsigned char* {
      return k == c ? stage + rt * kXRow : recv + (k * rpc + lr) * kXRow;
    };
    float M = -INFINITY;
#pragma unroll 1
    for (int k = 0; k < C; ++k) M = fmaxf(M, reinterpret_cast<const float*>(src(k) + 2 * D)[0]);
    const float mu = M == -INFINITY ? 0.f : M;
    float acc[16], L = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll 1
    for (int k = 0; k < C; ++k) {
      const unsigned char* r = src(k);
      const float mk = reinterpret_cast<const float*>(r + 2 * D)[0];
      if (mk != -INFINITY) {
        // w * l_k: the weight of the partial's normalised accumulator
        const float wl = fast_exp2(mk - mu) * reinterpret_cast<const float*>(r + 2 * D)[1];
        L += wl;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const uint2 h = *reinterpret_cast<const uint2*>(r + 2 * (4 * part + 32 * k4));
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
          acc[4 * k4] = fmaf(wl, a.x, acc[4 * k4]);
          acc[4 * k4 + 1] = fmaf(wl, a.y, acc[4 * k4 + 1]);
          acc[4 * k4 + 2] = fmaf(wl, b.x, acc[4 * k4 + 2]);
          acc[4 * k4 + 3] = fmaf(wl, b.y, acc[4 * k4 + 3]);
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __half* orow = p.out + (static_cast<long long>(seq) * p.num_q_heads + kvh * G + gg) * D;
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4)
      *reinterpret_cast<uint2*>(orow + 4 * part + 32 * k4) =
          make_uint2(pack_half2(acc[4 * k4] * inv, acc[4 * k4 + 1] * inv),
                     pack_half2(acc[4 * k4 + 2] * inv, acc[4 * k4 + 3] * inv));
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
  uint64_t* o_done = s_full + 6;               // one phase per sub-chunk's P V MMAs completed
  uint64_t* mma_done = s_full + 7;             // [2] every MMA of an issuer (S, PV) completed
  constexpr int kBars = 2 * NK + 2 * NV + 9;
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
  // Fused mode: after its nsub prefix sub-chunks the CTA attends the suffixes
  // (the table's columns past the prefix, W tokens per sequence) of the
  // sequences whose rows it finishes, [c * 128 / C, (c + 1) * 128 / C) of the
  // tile, as nsfx more sub-chunks: sub-chunk j holds a W-row segment for each
  // of the slice's sequences j * QPS .. j * QPS + QPS - 1 (QPS = 128 / W).
  // A sequence with s suffix tokens has them in the last s rows of its
  // segment (its blocks in reverse order, each copied from a token
  // coordinate shifted down so that the rows past its length fall before
  // the block and are filled with zeros by the copy), and each row takes only
  // its own segment's last s columns.
  const int P = p.prefix_blocks_n;
  const int W = FUSED ? (p.max_blocks - P) * BS : 0;  // 0, 16 or 32
  const int Wd = W > 0 ? W : kPfxTok;  // W as a divisor (only used when W > 0)
  const int QPS = kPfxTok / Wd;
  const int rpc = kPfxRows / static_cast<int>(gridDim.z);
  const int slice_s0 = (blockIdx.x * kPfxRows + c * rpc) / G;
  const int slice_n = W > 0 ? max(0, min(S, slice_s0 + rpc / G) - slice_s0) : 0;
  const int nsfx = (slice_n + QPS - 1) / QPS;
  const int ntot = nsub + nsfx;
  auto sub_len = [&](int t) {
    return t < nsub ? min(kPfxTok, tok_hi - (tok_lo + t * kPfxTok)) : kPfxTok;
  };
  // suffix tokens of a sequence of length L (checked against the prefix and
  // the table, a bad one reported when `report`)
  auto suffix_of = [&](int L, bool report) {
    const int cap = p.max_blocks * BS;
    if (L < P * BS || L > cap) {
      if (report) atomicOr(p.err, PA_DEVERR_BAD_LEN);
      L = L < 0 ? 0 : (L > cap ? cap : L);
    }
    return min(max(L - P * BS, 0), W);
  };

  if (threadIdx.x == 0) {
    // p_full counts the four softmax warps; the others one arrival (a TMA
    // transaction count or an MMA commit)
    for (int i = 0; i < kBars; ++i) {
      const bool softmax = &bars[i] >= p_full && &bars[i] < p_full + 2;
      mbar_init(smem_addr(&bars[i]), softmax ? kPfxSoftmaxWarps : 1);
    }
    *abort_flag = 0;
    if (FUSED) {
      // the other C - 1 chunks of the cluster each send this CTA the
      // partials of its rows (see the end of the kernel)
      const uint32_t rb = smem_addr(recv_bar);
      mbar_init(rb, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      mbar_arrive_expect_tx(rb, (gridDim.z - 1) * (kPfxRows / gridDim.z) * kXRow);
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
    // block id of slot `lane` of sub-chunk t, and (suffix sub-chunks) how
    // many of its rows are read: the copy's token coordinate is shifted down
    // by the rest, which the copy fills with zeros
    auto load_ids = [&](int t, int& valid) {
      const int nb = sub_len(t) / BS;
      int id = 0;
      valid = BS;
      if (lane < nb) {
        if (t < nsub) {
          id = __ldg(p.prefix_blocks + (tok_lo + t * kPfxTok) / BS + lane);
          if (id < 0 || id >= p.num_blocks) {
            if (is_k) atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
            id = 0;  // an in-range block keeps the byte count; the result is flagged
          }
        } else {
          // suffix sub-chunk: slot `lane` holds block jb of the slice's
          // sequence q, the segment's blocks in reverse order
          const int bpq = Wd / BS, q = (t - nsub) * QPS + lane / bpq;
          const int jb = bpq - 1 - lane % bpq;
          valid = 0;
          if (q < slice_n) {
            const int seq = slice_s0 + q;
            const int v = min(max(suffix_of(p.seq_lens[seq], false) - jb * BS, 0), BS);
            if (v > 0) {
              id = p.block_table[static_cast<long long>(seq) * p.max_blocks + P + jb];
              if (id < 0 || id >= p.num_blocks) {
                if (is_k) atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
                id = 0;
              } else {
                valid = v;
              }
            }
          }
          // a slot with no rows read copies only fill (zeros)
        }
      }
      return id;
    };
    int next_valid = BS;
    int next_ids = ntot > 0 ? load_ids(0, next_valid) : 0;
    for (int t = 0; t < ntot; ++t, ++issued) {
      const int st = t % nst, n = sub_len(t);
      const int ids = next_ids, valids = next_valid;
      if (t >= nst &&
          !warp_wait_phase(smem_addr(&empty[st]), ((t / nst) - 1) & 1, abort_flag, p.err))
        break;
      const uint32_t dst = smem_addr(ring + st * kPfxTile), bar = smem_addr(&full[st]);
      if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * 256u);
      for (int j = 0; j < n / BS; ++j) {
        const int phys = __shfl_sync(0xffffffffu, ids, j);
        const int y0 = __shfl_sync(0xffffffffu, valids, j) - BS;  // 0 but in suffix slots
        if (lane == 0) {
#pragma unroll
          for (int sb = 0; sb < BS / 16; ++sb) {
            const uint32_t off = static_cast<uint32_t>(j * BS + sb * 16) * 128u;
            tma_load_4d(dst + off, map, 0, y0 + sb * 16, kvh, phys, bar);
            tma_load_4d(dst + HALF + off, map, 64, y0 + sb * 16, kvh, phys, bar);
          }
        }
      }
      if (t + 1 < ntot) next_ids = load_ids(t + 1, next_valid);
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
    for (int t = 0; t < ntot; ++t) {
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
    // ---- PV issuer: O += P_t V_t, O in TMEM for the whole chunk ----
    for (int t = 0; t < ntot; ++t) {
      const int st = t % NV, b = t & 1;
      if (!warp_wait_phase(smem_addr(&p_full[b]), (t >> 1) & 1, abort_flag, p.err)) break;
      if (!warp_wait_phase(smem_addr(&v_full[st]), (t / NV) & 1, abort_flag, p.err)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t vb = smem_addr(v_s + st * kPfxTile);
        const uint32_t id = f16_idesc(D, true);
        const int n = sub_len(t);
        // A = P over S buffer b: 16 tokens per MMA, 8 TMEM columns
        for (int k = 0; k < n / 16; ++k)
          tc_mma_ts(tmem + kPfxOCol, tmem + b * kPfxTok + 8 * k,
                    sw128_desc(vb + k * 2048, HALF, 1024), id, (t > 0 || k > 0) ? 1u : 0u);
        tc_commit(smem_addr(o_done));
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
    const int r = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t o_tm = lane_base + kPfxOCol;
    // scores are scaled by qscale (any sign); the row max of the scaled
    // scores is the max of the raw ones times qscale, or the min if qscale < 0
    const bool qpos = p.qscale >= 0.f;
    // fused mode: this row's place among the slice's sequences (-1: not in
    // the slice) and its sequence's length, read now and checked when the
    // suffix sub-chunks come
    int sfx_q = -1, sfx_len = 0;
    if (FUSED && r >= c * rpc && r < (c + 1) * rpc) {
      const int seq = (blockIdx.x * kPfxRows + r) / G;
      if (seq < S) {
        sfx_q = seq - slice_s0;
        sfx_len = p.seq_lens[seq];
      }
    }
    float m = -INFINITY, l = 0.f;
    bool ok = true, arrived = false;
    for (int t = 0; t < ntot; ++t) {
      const int n = sub_len(t), b = t & 1;
      if (!warp_wait_phase(smem_addr(&s_full[b]), (t >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      if (FUSED && t == ntot - 1) {
        // this CTA's last S MMAs have completed: its Q and K tiles are free
        // for the rows the cluster sends it (see below)
        cluster_arrive();
        arrived = true;
      }
      tc_fence_after();
      const uint32_t sa = lane_base + b * kPfxTok;
      uint32_t sv[kPfxTok];
      tmem_ld128(sa, sv);
      const uint32_t neutral = qpos ? 0xff800000u : 0x7f800000u;  // -inf / +inf
      if (n < kPfxTok) {
        // a short last sub-chunk: the columns past it hold no scores; they
        // take no part in the max, their P is never read (the P V MMAs stop
        // at n) and their sum is left out below
#pragma unroll
        for (int i = 0; i < kPfxTok; ++i)
          if (i >= n) sv[i] = neutral;
      }
      if (FUSED && t >= nsub) {
        // a suffix sub-chunk: this row's columns are the last s of its own
        // sequence's segment; every other score becomes the neutral value,
        // whose P is exactly 0 (qscale is not 0 here)
        const int j = t - nsub;
        const bool mine = sfx_q >= j * QPS && sfx_q < (j + 1) * QPS;
        const int hi = mine ? (sfx_q - j * QPS + 1) * W : 0;
        const int lo = mine ? hi - suffix_of(sfx_len, (blockIdx.x * kPfxRows + r) % G == 0) : 0;
#pragma unroll
        for (int i = 0; i < kPfxTok; ++i)
          if (i < lo || i >= hi) sv[i] = neutral;
      }
      float e4[4];
      if (qpos) {
        e4[0] = e4[1] = e4[2] = e4[3] = -INFINITY;
#pragma unroll
        for (int i = 0; i < kPfxTok; ++i) e4[i & 3] = fmaxf(e4[i & 3], __uint_as_float(sv[i]));
      } else {
        e4[0] = e4[1] = e4[2] = e4[3] = INFINITY;
#pragma unroll
        for (int i = 0; i < kPfxTok; ++i) e4[i & 3] = fminf(e4[i & 3], __uint_as_float(sv[i]));
      }
      const float ext = qpos ? fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3]))
                             : fminf(fminf(e4[0], e4[1]), fminf(e4[2], e4[3]));
      const float mx = ext * p.qscale;
      // The reference max m moves only when this sub-chunk's max exceeds it
      // by more than kRescaleLog2; otherwise P is taken against m (each
      // value at most 2^kRescaleLog2) and O in TMEM is left as it is.
      const bool grow = mx > m + kRescaleLog2;
      if (t > 0 && __any_sync(0xffffffffu, grow)) {
        // O holds P V up to the previous sub-chunk once those MMAs complete
        // (S_t was issued after P V of sub-chunk t - 2 had completed, so
        // o_done is at most one phase short of the one waited for)
        if (!warp_wait_phase(smem_addr(o_done), (t - 1) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = grow ? fast_exp2(m - mx) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float v[32];
          tmem_ld32(o_tm + c0, v);
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i] * f);
          tmem_st32(o_tm + c0, w);
        }
      }
      if (grow) {
        l *= fast_exp2(m - mx);  // 0 while m is -inf
        m = mx;
      }
      // P = exp2(S * qscale - m) as fp16 pairs, written over the S columns:
      // tokens 2i, 2i+1 go to column i; sums per 16 tokens. While m is still
      // -inf every score so far was masked: take 0, so that masked scores
      // give exactly 0 (not NaN)
      const float mz = m == -INFINITY ? 0.f : m;
      uint32_t h[kPfxTok / 2];
      float sum16[kPfxTok / 16];
#pragma unroll
      for (int g = 0; g < kPfxTok / 16; ++g) sum16[g] = 0.f;
#pragma unroll
      for (int i = 0; i < kPfxTok / 2; ++i) {
        const float e0 = fast_exp2(fmaf(__uint_as_float(sv[2 * i]), p.qscale, -mz));
        const float e1 = fast_exp2(fmaf(__uint_as_float(sv[2 * i + 1]), p.qscale, -mz));
        sum16[i / 8] += e0 + e1;
        h[i] = pack_half2(e0, e1);
      }
      tmem_st64(sa, h);
      float sum = 0.f;
#pragma unroll
      for (int g = 0; g < kPfxTok / 16; ++g) sum += g * 16 < n ? sum16[g] : 0.f;
      l += sum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&p_full[b]));
    }
    // a table with no columns past the prefix: each length must be the prefix's
    if (FUSED && W == 0 && sfx_q >= 0) suffix_of(sfx_len, (blockIdx.x * kPfxRows + r) % G == 0);
    if (FUSED && !arrived) cluster_arrive();
    // O (relative to m) once every P V MMA has completed: the PV issuer's
    // final commit (o_done cannot tell: up to two of its phases may still be
    // open here)
    if (ok && ntot > 0) {
      ok = warp_wait_phase(smem_addr(&mma_done[1]), 0, abort_flag, p.err);
      if (ok) tc_fence_after();
    }
    constexpr int kPad = D + 4;
    if constexpr (FUSED) {
      // The row's partial, staged in this CTA's V tiles (free: every P V MMA
      // has completed) as kXRow bytes: the accumulator divided by the sum as
      // fp16 (within the range of the V values it averages), then max and
      // sum; the warp then copies its rows of each other CTA's slice into
      // that CTA's Q and K tiles, free once every CTA has arrived above.
      unsigned char* srow = v_s + r * kXRow;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        if (ok && ntot > 0) {
          tmem_ld32(o_tm + c0, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          *reinterpret_cast<uint4*>(srow + 2 * (c0 + i)) =
              make_uint4(pack_half2(v[i] * inv_l, v[i + 1] * inv_l),
                         pack_half2(v[i + 2] * inv_l, v[i + 3] * inv_l),
                         pack_half2(v[i + 4] * inv_l, v[i + 5] * inv_l),
                         pack_half2(v[i + 6] * inv_l, v[i + 7] * inv_l));
      }
      *reinterpret_cast<float2*>(srow + 2 * D) = make_float2(m, l);
      fence_proxy_async_smem();
      __syncwarp();
      cluster_wait();
      if (lane == 0) {
        // rows 32 * warp .. + 31 split by the slice they belong to
        const int C = static_cast<int>(gridDim.z);
        for (int k = (warp * 32) / rpc; k <= (warp * 32 + 31) / rpc && k < C; ++k) {
          if (k == c) continue;
          const int r0 = max(warp * 32, k * rpc), r1 = min(warp * 32 + 32, (k + 1) * rpc);
          bulk_copy_s2cluster(
              cluster_map(smem_addr(q_s) + static_cast<uint32_t>((c * rpc + r0 - k * rpc) * kXRow),
                          k),
              smem_addr(v_s) + static_cast<uint32_t>(r0 * kXRow),
              static_cast<uint32_t>((r1 - r0) * kXRow), cluster_map(smem_addr(recv_bar), k));
        }
      }
    } else {
      // Every MMA has completed, so the K tiles are free: each warp stages its
      // rows there (16.5 KB, rows padded to 132 floats against bank
      // conflicts) and writes each sequence's G rows as one contiguous run
      float* stage = reinterpret_cast<float*>(k_s) + warp * 32 * kPad;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        if (ok && ntot > 0) {
          tmem_ld32(o_tm + c0, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(stage + lane * kPad + c0 + i) =
              make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      }
      __syncwarp();
      const int row = blockIdx.x * kPfxRows + r, seq = row / G, gg = row % G;
      const bool write = ok && !*abort_flag;
      if (seq < S && write) {
        float* rec =
            p.records + ((static_cast<long long>(c) * S + seq) * p.num_kv_heads + kvh) * RS;
        rec[G * D + 2 * gg] = m;
        rec[G * D + 2 * gg + 1] = l;
      }
      if (write) {
        // the warp's rows 32w .. 32w+31 belong to sequences row / G; a
        // record's G rows are contiguous ([G][D] floats)
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
  }
  // Fused mode: every thread of every CTA of the cluster (the chunks of this
  // row tile and KV head) arrives once on the barrier the softmax warps wait
  // for before sending rows, whatever happened before: the softmax warps
  // when their last S has been read, the other warps after their loops.
  if constexpr (FUSED) {
    if (warp >= kPfxSoftmaxWarps) cluster_arrive();
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
    if (warp >= kPfxSoftmaxWarps) cluster_wait();
    fused_merge<G>(p, v_s, q_s, recv_bar, kvh, c);
    // the barrier fused_merge arrived on: every CTA's rows have landed where
    // they were sent, so no copy out of a CTA's shared memory is still
    // running when it leaves
    cluster_wait();
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
  pp.out = static_cast<__half*>(call.out);
  pp.max_blocks = call.max_blocks;
  const int S = call.num_seqs, Hkv = call.num_kv_heads, P = call.prefix_blocks_n;
  // One launch when every suffix is short, the clusters fit and each CTA's
  // suffixes fill at most kMaxSuffixSub sub-chunks. The suffix masks need
  // qscale != 0 (a zero scale makes every weight equal: the unfused path
  // handles it).
  const int W = (call.max_blocks - P) * BS;
  if (W <= kFusedSuffixTokens && call.qscale != 0.f) {
    const PfxGeom fg = fused_prefix_geometry(S, G, Hkv, P, dev.sm_count);
    const int per_slice = kPfxRows / fg.chunks / G;  // sequences whose rows one CTA finishes
    const int nsfx = (per_slice * W + kPfxTok - 1) / kPfxTok;
    if (nsfx <= kMaxSuffixSub && fused_prefix_fits<BS, G>(fg, dev)) {
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
