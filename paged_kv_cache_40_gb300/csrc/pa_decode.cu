// Paged decode attention for GB300 (sm_103a).
//
// What it computes ("Phase 7 · Document 04 — PagedAttention", §2 Core
// Concept; lux-666 notes "PagedAttention", 最小模型): for every sequence i and
// query head h, the softmax-weighted sum of the V rows of its cached tokens,
// with weights softmax(scale * q[i][h] . K[t]); the K/V rows of token t are
// found through the sequence's block table: physical block
// block_table[i][t / BS], row t % BS, KV head h / G.
//
// How (GB300-first; the pages give no kernel, only the layout sketch):
//   * Head groups. A CTA streams HG KV heads of a block together (HG = the
//     largest of 8, 4, 2, 1 dividing the KV head count). For the common 8-KV-
//     head models that is the whole block: one contiguous 32 KB region of K
//     and one of V per 16-token block, moved by four 16 KB TMA copies, which
//     keeps DRAM pages and the copy engine efficient. One consumer warp owns
//     one KV head of the group and all G query heads that read it (GQA
//     head-group reuse: every K/V byte is read from HBM once per step).
//   * Segments and balanced chunks. A segment is (sequence, head group): the
//     ceil(L/BS) blocks of that group. Segments are laid end to end (sequence-
//     major) into one stream of blocks, and the stream is cut into equal
//     contiguous chunks, one per CTA of a persistent grid (SMs x resident
//     CTAs): every CTA streams the same number of blocks. A segment inside one
//     chunk is finished there and each warp writes its head's output straight
//     from registers. A segment cut by chunk boundaries leaves one partial
//     result per (chunk, head); the last warp to finish a head merges that
//     head's partials with the log-sum-exp rule. It learns that it is last
//     from an arrival counter per (sequence, KV head), taken with a
//     compare-and-swap, never a spin: the counter word carries a tag unique
//     to the call next to the count, so a word left by an earlier call (or
//     never written) counts as zero arrivals and the workspace needs no
//     clearing. A chunk has at most two cut pieces, its first and its last;
//     each CTA streams them before the uncut segments in between, so most
//     merges happen while the other CTAs are still streaming.
//   * Warp specialisation. A producer warp is the only one that walks the
//     CTA's chunk, finding a stream position's segment with a warp-wide
//     32-way search over the prefix sums. It loads the block-table entries of
//     the next 32 blocks while it issues the current ones (and uses them only
//     after), and moves K and V with TMA into a
//     ring of shared-memory stages: a 4-D tensor map over the pool seen as
//     (dim, token, KV head, block) — token stride larger than head stride —
//     with box {64, tokens, HG, 1} and the 128-byte swizzle, so each head's
//     rows land contiguously and the tensor-core fragment loads (ldmatrix)
//     are free of bank conflicts. Every consumer warp reads every stage (its
//     own head), so a stage is released after HG arrivals. For each piece the
//     producer also publishes, in one of two q slots, the piece's metadata
//     and its q rows, so the next piece's q is in flight while the current
//     one streams and the consumers never search the block stream. For fp16
//     pools the copies carry an L2 evict-first policy: the stream is read once,
//     and what is read again (partial records, counters, table, q, the code)
//     stays in L2 while it passes.
//     Merge warps take the cut pieces off the consumers' critical path: the
//     consumer warps write their partial records, send a message (segment and
//     place) through a small shared-memory ring and go on streaming; the
//     merge warps count the arrivals of all HG heads at once (one lane each)
//     and merge the heads whose partials are complete. Only the CTA's final
//     piece is merged by the consumer warps themselves, in parallel.
//   * Consumer math on tensor cores (mma.sync m16n8k16, fp16 in, fp32
//     accumulate). Scores S = Q K^T with the G query heads as the M rows and
//     8-token groups as N; the online softmax (base 2, running max and sum)
//     works on the accumulator registers; then O^T += V^T P^T with head_dim as
//     M and the heads as N, whose B operand is exactly the probabilities the
//     score accumulators already hold (no transpose, no shared-memory trip).
//     Rows past the sequence end are masked out of the softmax and zeroed in
//     the V stage so they contribute exactly nothing.
//   * Programmatic dependent launch: the CTAs may start while the previous
//     kernel on the stream finishes, set up their barriers and ask L2 for the
//     lengths, the table and q, but read no input before that kernel has
//     completed (griddepcontrol.wait), so it may write any of them.
//   * Every wait is bounded (about one second of %globaltimer); on expiry the
//     kernel records PA_DEVERR_TIMEOUT, stops issuing copies, drains the copies
//     already in flight (again bounded) and finishes without faulting.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tma.h"

namespace {

constexpr int kMaxHG = 8;                          // KV heads per group = consumer warps
constexpr int kMergeWarps = 3;                     // warps merging cut pieces off the stream
constexpr int kMaxThreads = (kMaxHG + 1 + kMergeWarps) * 32;  // consumers, producer, mergers
constexpr int kMsgSlots = 4;                       // cut pieces in flight to the merge warps
constexpr int kMaxSeqs = 16384;
constexpr int kMaxGrid = 1024;
constexpr int kMaxStages = 16;
constexpr int kRingBytesPerHead = 24 * 1024;       // ring size per KV head of the group
constexpr int kArrivalBits = 20;                   // low bits of a counter word: arrivals
constexpr long long kPrefetchLines = 1ll << 17;     // 16 MB of table and q asked of L2 at most

// ------------------------------------------------------------- shapes ---

// KV heads a CTA streams together: the largest of 8, 4, 2, 1 dividing Hkv.
__host__ __device__ constexpr int head_group(int hkv) {
  return hkv % 8 == 0 ? 8 : hkv % 4 == 0 ? 4 : hkv % 2 == 0 ? 2 : 1;
}

template <int D, int BS, int G, bool KV8 = false>
struct Shape {
  static_assert(G >= 1 && G <= 8, "at most 8 query heads per KV head (mma N = 8)");
  static_assert(D % 64 == 0 && BS % 8 == 0, "shape");
  static_assert(!KV8 || (D == 128 && BS >= 16), "fp8 pools: head_dim 128, 16-token stages");
  static constexpr int ESZ = KV8 ? 1 : 2;            // bytes per cached value
  static constexpr int NHALF = D * ESZ / 128;        // 128-byte lines per row
  static constexpr int TS = BS < 16 ? BS : 16;       // tokens per stage
  static constexpr int REC = rec_floats(G, D);
  // shared-memory layout: fixed part (bytes)
  static constexpr int OFF_FULL = 0;
  static constexpr int OFF_EMPTY = OFF_FULL + kMaxStages * 8;
  static constexpr int OFF_QFULL = OFF_EMPTY + kMaxStages * 8;   // [2]
  static constexpr int OFF_QEMPTY = OFF_QFULL + 2 * 8;            // [2]
  static constexpr int OFF_MFULL = OFF_QEMPTY + 2 * 8;            // [kMsgSlots]
  static constexpr int OFF_MEMPTY = OFF_MFULL + kMsgSlots * 8;    // [kMsgSlots]
  static constexpr int OFF_PMETA = OFF_MEMPTY + kMsgSlots * 8;    // PieceMeta [2]
  static constexpr int OFF_MMETA = OFF_PMETA + 2 * 64;            // MsgMeta [kMsgSlots]
  static constexpr int OFF_FLAGS = OFF_MMETA + kMsgSlots * 32;    // 32 ints, see kFlag*
  static constexpr int FIXED = OFF_FLAGS + 128;
  static int stage_bytes(int hg) { return 2 * NHALF * hg * TS * 128; }
  // then, from the next 1 KB-aligned address (the swizzle pattern is a
  // function of address bits 7..9): ring, two q slots, prefix
  static size_t smem_bytes(int hg, int nst, int num_seqs) {
    return static_cast<size_t>(FIXED) + 1024 + static_cast<size_t>(nst) * stage_bytes(hg) +
           2 * static_cast<size_t>(hg) * G * D * 2 + static_cast<size_t>(num_seqs + 1) * 4;
  }
};

// int flags in shared memory
constexpr int kFlagAbort = 0;   // set when a bounded wait gave up
constexpr int kFlagWsum = 8;    // [12] warp sums of the prefix scan

struct DecodeParams {
  const __half* q;
  const __half* k_pool;
  const __half* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  __half* out;
  const float* k_scale;  // fp8 pools: [num_kv_heads] dequantization scales (else unused)
  const float* v_scale;
  float* records;  // [2 * max_chunks][HG][rec_floats(G, D)] partials of cut segments
  unsigned long long* counters;  // [num_seqs][num_kv_heads] (tag << kArrivalBits) | arrivals
  unsigned long long tag;        // this call's tag, nonzero, < 2^(64 - kArrivalBits)
  int32_t* err;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int max_blocks;
  int num_blocks;
  int cap_blocks;  // max blocks per chunk (0 = balance over the grid)
  // shared-prefix mode: the table pointer starts past the prefix's
  // pfx_blocks columns, lengths count past its pfx_blocks * BS tokens, and
  // every result also folds the pfx_chunks prefix records of its (sequence,
  // KV head), record index pfx_rec_base + (chunk * S + seq) * Hkv + kvh
  int pfx_blocks;
  int pfx_chunks;
  long long pfx_rec_base;
  long long pfx_own_base;  // [S][Hkv] records of segments streamed whole
  int hg;          // KV heads per group (consumer warps)
  int nst;         // ring stages
  float qscale;    // scale * log2(e)
  unsigned long long wait_ns;    // time limit of the pipeline waits
  long long block_stride_bytes;  // host only: the pools' block stride, for their tensor maps
  // append mode (fp16 pools, not shared-prefix mode): each sequence's new K/V
  // row (k_new/v_new [num_seqs][num_kv_heads][D]) goes to slot_mapping[seq],
  // which must be the row of its last token; the producer writes it just
  // before it copies that block, so the attention sees it
  const __half* k_new;
  const __half* v_new;
  const int32_t* slot_mapping;
  long long block_stride;        // values from one pool block to the next
};

__device__ __forceinline__ int clamp_len(int L, int cap, int32_t* err) {
  if (L < 0 || L > cap) {
    atomicOr(err, PA_DEVERR_BAD_LEN);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

// Blocks per sequence -> exclusive prefix sum pfx[0..S] in shared memory,
// computed by all threads of the block (wsum: one int per warp). Lengths
// outside [0, cap] are clamped and reported.
__device__ __forceinline__ void block_prefix(int* pfx, int* wsum, const int32_t* seq_lens, int S,
                                             int bs, int cap, int32_t* err, int len_off = 0) {
  const int tid = threadIdx.x, nthreads = blockDim.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < S; i += nthreads) {
    const int Lfull = __ldg(seq_lens + i);
    if (Lfull < len_off) atomicOr(err, PA_DEVERR_BAD_LEN);  // shorter than a shared prefix
    const int L = clamp_len(max(Lfull - len_off, 0), cap, err);
    pfx[i + 1] = (L + bs - 1) / bs;
  }
  if (tid == 0) pfx[0] = 0;
  __syncthreads();
  const int per = (S + nthreads - 1) / nthreads;
  const int lo = min(S, tid * per), hi = min(S, lo + per);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += pfx[i + 1];
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int run = incl - sum;
  for (int w = 0; w < warp; ++w) run += wsum[w];
  for (int i = lo; i < hi; ++i) {
    run += pfx[i + 1];
    pfx[i + 1] = run;
  }
  __syncthreads();
}

// The block stream cut into chunks: one per CTA (or of at most cap_blocks
// blocks each, a CTA then taking every gridDim.x-th chunk). Stream positions
// fit in 32 bits (the host checks num_seqs x head groups x max blocks).
struct Geometry {
  int total, chunk, nchunks;
};
__device__ __forceinline__ Geometry chunk_geometry(int total, int grid, int cap_blocks) {
  Geometry g;
  g.total = total;
  g.chunk = (total + grid - 1) / grid;
  if (cap_blocks > 0 && g.chunk > cap_blocks) g.chunk = cap_blocks;
  if (g.chunk < 1) g.chunk = 1;
  g.nchunks = (total + g.chunk - 1) / g.chunk;
  return g;
}

// Record of chunk cc for a segment starting at stream index s0 whose first
// chunk is c_first: slot 0 if the segment covers the chunk's start (the
// chunk's first piece), slot 1 if it begins inside the chunk.
__device__ __forceinline__ long long record_index(int cc, int c_first, int s0, int chunk, int hg,
                                                  int w) {
  return static_cast<long long>(2 * cc + ((cc == c_first && s0 > cc * chunk) ? 1 : 0)) * hg + w;
}

// The K/V stream is read once per launch: for fp16 pools its TMA copies
// carry an L2 evict-first policy, so the lines they bring in are the first
// to go and what the CTAs read again (partial records, counters, table, q,
// the code) stays in L2 while hundreds of megabytes stream past. (On 64
// sequences of 128 to 2048 tokens, 8 KV heads of 128 dims, 302 MB a launch,
// that took 1.6 us off 57.7 us; the half-size E4M3 stream measured 0.25 us
// slower with it, so fp8 pools copy without it.)
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_4d_once(uint32_t dst, const CUtensorMap* map, int x,
                                                 int y, int z, int w, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(pol)
      : "memory");
}

// Position in the block stream -> (sequence, head group, block within segment).
struct Cursor {
  int seq, hg, j, nb;  // nb = blocks in the segment (sequence)
  int seg_start;       // stream index of the segment's block 0
};

// Called by a whole warp (all 32 lanes, same x): the sequence is found by a
// 32-way search, each lane probing one of 32 evenly spaced prefix entries,
// so S sequences take ceil(log32 S) rounds of one shared-memory load each.
__device__ __forceinline__ Cursor locate(int x, const int* pfx, int S, int nhg) {
  const int lane = threadIdx.x & 31;
  int lo = 0, n = S;  // the largest i with pfx[i] * nhg <= x lies in [lo, lo + n)
  while (n > 1) {
    const int step = (n + 31) >> 5;
    const int idx = lo + lane * step;
    const unsigned le = __ballot_sync(0xffffffffu, idx < lo + n && pfx[idx] * nhg <= x);
    const int k = 31 - __clz(le);  // lane 0's probe is pfx[lo], always <= x
    lo += k * step;
    n = min(step, n - k * step);
  }
  Cursor c;
  c.seq = lo;
  c.nb = pfx[lo + 1] - pfx[lo];
  const int r = x - pfx[lo] * nhg;
  c.hg = r / c.nb;
  c.j = r - c.hg * c.nb;
  c.seg_start = pfx[lo] * nhg + c.hg * c.nb;
  return c;
}


// Pieces of chunk c in the order a CTA streams them: the piece at the chunk's
// start, then the piece at its end if that one's segment runs past the chunk,
// then the uncut segments in between. Both cut pieces (whose partials other
// chunks wait for) are thus finished early. Only the producer walks; the
// other warps learn each piece from it.
struct Walk {
  int c;       // chunk
  int x0, xe;  // chunk [x0, xe) of the block stream
  int x1;      // end of the first piece
  int xl;      // start of the trailing cut piece (xe if there is none)
  int xm;      // next uncut segment
  int phase;   // 0: first piece next, 1: trailing cut piece next, 2: middle
  Cursor first, last;  // cursors at x0 and at xl
};

__device__ __forceinline__ void walk_begin(Walk& wk, int c, const Geometry& geo, const int* pfx,
                                           int S, int nhg) {
  wk.c = c;
  wk.phase = 0;
  if (c >= geo.nchunks) return;
  wk.x0 = c * geo.chunk;
  wk.xe = min(geo.total, wk.x0 + geo.chunk);
  wk.first = locate(wk.x0, pfx, S, nhg);
  wk.x1 = min(wk.first.seg_start + wk.first.nb, wk.xe);
  wk.xl = wk.xe;
  if (wk.x1 < wk.xe) {
    wk.last = locate(wk.xe - 1, pfx, S, nhg);
    if (wk.last.seg_start + wk.last.nb > wk.xe) {
      wk.xl = wk.last.seg_start;
      wk.last.j = 0;
    }
  }
  wk.xm = wk.x1;
}

// A piece: cursor at its first block, n blocks, and its chunk.
struct Piece {
  Cursor cur;
  int n, c;
};

// Next piece of the walk, moving on to the CTA's next chunk (c + stride) when
// this one is done. False at the end.
__device__ __forceinline__ bool walk_next(Walk& wk, const Geometry& geo, int stride,
                                          const int* pfx, int S, int nhg, Piece& pc) {
  while (wk.c < geo.nchunks) {
    pc.c = wk.c;
    if (wk.phase == 0) {
      wk.phase = 1;
      pc.cur = wk.first;
      pc.n = wk.x1 - wk.x0;
      return true;
    }
    if (wk.phase == 1) {
      wk.phase = 2;
      if (wk.xl < wk.xe) {
        pc.cur = wk.last;
        pc.n = wk.xe - wk.xl;
        return true;
      }
    }
    if (wk.xm < wk.xl) {
      pc.cur = locate(wk.xm, pfx, S, nhg);
      pc.n = min(pc.cur.nb - pc.cur.j, wk.xl - wk.xm);
      wk.xm += pc.n;
      return true;
    }
    walk_begin(wk, wk.c + stride, geo, pfx, S, nhg);
  }
  return false;
}

// What the producer tells the other warps about a piece (in shared memory,
// published by the arrival on the piece's q slot barrier).
struct PieceMeta {
  int seq, hg, j, n, nb, len, s0, c, last, pad[7];
};
// A cut piece handed from the consumer warps to the merge warps.
struct MsgMeta {
  int seq, hg, nb, s0, stop, pad[3];
};

// Counts one arrival of a cut segment's head on its tagged counter word and
// returns true for the arrival that completes the count (E >= 2 arrivals),
// which also puts the word back to zero so that a later call, even one with
// the same tag (a replayed launch), starts from no arrivals. A word whose tag
// is not this call's (zero, or left by an earlier call) counts as none: the
// first arrival installs the tag with a compare-and-swap from `seen`, the
// caller's guess of the word (0 if it has none; retried from the value each
// failure returns, until the tag is there). Every other arrival is one
// atomic add, a single round trip to L2 whatever the others do.
__device__ __forceinline__ bool arrive_last(unsigned long long* word, unsigned long long tag,
                                            unsigned E, unsigned long long seen, int32_t* err) {
  constexpr unsigned long long kCountMask = (1ull << kArrivalBits) - 1;
  if ((seen >> kArrivalBits) != tag) {
    for (int i = 0;; ++i) {
      if (i == 4096) {
        atomicOr(err, PA_DEVERR_TIMEOUT);
        return false;
      }
      const unsigned long long got = atomicCAS(word, seen, (tag << kArrivalBits) | 1ull);
      if (got == seen) return false;  // the first of E >= 2 arrivals
      if ((got >> kArrivalBits) == tag) break;
      seen = got;
    }
  }
  const unsigned long long old = atomicAdd(word, 1ull);
  if ((old >> kArrivalBits) != tag || (old & kCountMask) + 1 > E) {
    atomicOr(err, PA_DEVERR_TIMEOUT);  // cannot happen: the tag stays until the count is full
    return false;
  }
  if ((old & kCountMask) + 1 < E) return false;
  // the last arrival: no other arrival of this call is left to touch the word
  *reinterpret_cast<volatile unsigned long long*>(word) = 0ull;
  return true;
}

// Shared-prefix mode: wait for the prefix kernel (the grid launched just
// before on the stream) before reading its records.
template <bool PFX>
__device__ __forceinline__ void pfx_wait() {
  if constexpr (PFX) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// One warp merges the E partial records of one KV head of a cut segment with
// the log-sum-exp rule and writes that head's G fp16 output rows. Record i is
// `recs + rec_of(i) * rec_floats(G, D)`: acc [G][D], then (max, sum) per
// head. Records are folded in batches of KB: lane r*G + h loads the (max,
// sum) of record r, head h, and every lane loads its float4 slices (l,
// l + 32, ...) of each record's accumulator; a slice lies inside one query
// head, whose (max, sum) the lane then takes by shuffle. All loads of a batch
// are issued before any is used, so a batch costs one L2 round trip.
template <int D, int G, typename RecOf>
__device__ __forceinline__ void merge_partials(const float* recs, int E, RecOf rec_of,
                                               __half* out_row) {
  constexpr int NV4 = G * D / 4;         // float4 slices of one accumulator
  constexpr int PER = (NV4 + 31) / 32;   // slices per lane
  // records per batch: (max, sum) pairs fit one per lane, and the slices in
  // flight stay within registers
  constexpr int KB_ML = 32 / G;
  constexpr int KB_REG = PER >= 8 ? 2 : 20 / PER;
  constexpr int KB = KB_ML < KB_REG ? KB_ML : KB_REG;
  constexpr int RS = rec_floats(G, D);   // floats per record (16-byte multiple)
  const int lane = threadIdx.x & 31;
  float M[PER], Ls[PER];
  float4 A[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    M[k] = -INFINITY;
    Ls[k] = 0.f;
    A[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int base = 0; base < E; base += KB) {
    float2 mlv = make_float2(-INFINITY, 0.f);
    {
      const int r = lane / G, h = lane % G;
      if (r < KB && base + r < E)
        mlv = __ldcg(reinterpret_cast<const float2*>(recs + rec_of(base + r) * RS + G * D) + h);
    }
    float4 v[KB][PER];
#pragma unroll
    for (int r = 0; r < KB; ++r) {
      const bool have = base + r < E;
      const float* rp = recs + (have ? rec_of(base + r) : 0) * RS;
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i = lane + 32 * k;
        v[r][k] = have && i < NV4 ? __ldcg(reinterpret_cast<const float4*>(rp) + i)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = lane + 32 * k;
      const int hk = i < NV4 ? (i * 4) / D : 0;
      float mr[KB], lr[KB];
#pragma unroll
      for (int r = 0; r < KB; ++r) {
        mr[r] = __shfl_sync(0xffffffffu, mlv.x, r * G + hk);
        lr[r] = __shfl_sync(0xffffffffu, mlv.y, r * G + hk);
      }
      float mb = M[k];
#pragma unroll
      for (int r = 0; r < KB; ++r) mb = fmaxf(mb, mr[r]);
      const float mu = mb == -INFINITY ? 0.f : mb;
      const float f = fast_exp2(M[k] - mu);
      float4 a = make_float4(A[k].x * f, A[k].y * f, A[k].z * f, A[k].w * f);
      float l = Ls[k] * f;
#pragma unroll
      for (int r = 0; r < KB; ++r) {
        const float wr = fast_exp2(mr[r] - mu);
        a.x += v[r][k].x * wr;
        a.y += v[r][k].y * wr;
        a.z += v[r][k].z * wr;
        a.w += v[r][k].w * wr;
        l += lr[r] * wr;
      }
      A[k] = a;
      Ls[k] = l;
      M[k] = mb;
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = lane + 32 * k;
    if (i < NV4) {
      const float inv = Ls[k] > 0.f ? 1.f / Ls[k] : 0.f;
      __half2* o = reinterpret_cast<__half2*>(out_row + i * 4);
      o[0] = __floats2half2_rn(A[k].x * inv, A[k].y * inv);
      o[1] = __floats2half2_rn(A[k].z * inv, A[k].w * inv);
    }
  }
}

template <int D, int BS, int G, bool KV8, bool PFX = false>
__global__ void __launch_bounds__(kMaxThreads, 1)
    paged_decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  using SH = Shape<D, BS, G, KV8>;
  constexpr int TS = SH::TS;
  constexpr int QBYTES_PER_HEAD = G * D * 2;
  extern __shared__ __align__(128) unsigned char smem[];
  const int HG = p.hg, NST = p.nst;
  const int HALF = HG * TS * 128;        // one 64-dim half of one stage's K (or V)
  const int TILE = SH::NHALF * HALF;     // K (or V) of one stage
  const int STAGE = 2 * TILE;
  const int QSLOT = HG * QBYTES_PER_HEAD;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + SH::OFF_FULL);
  uint64_t* empty_bar = reinterpret_cast<uint64_t*>(smem + SH::OFF_EMPTY);
  uint64_t* qfull_bar = reinterpret_cast<uint64_t*>(smem + SH::OFF_QFULL);
  uint64_t* qempty_bar = reinterpret_cast<uint64_t*>(smem + SH::OFF_QEMPTY);
  uint64_t* mfull_bar = reinterpret_cast<uint64_t*>(smem + SH::OFF_MFULL);
  uint64_t* mempty_bar = reinterpret_cast<uint64_t*>(smem + SH::OFF_MEMPTY);
  PieceMeta* pmeta = reinterpret_cast<PieceMeta*>(smem + SH::OFF_PMETA);
  MsgMeta* mmeta = reinterpret_cast<MsgMeta*>(smem + SH::OFF_MMETA);
  int* flags = reinterpret_cast<int*>(smem + SH::OFF_FLAGS);
  volatile int* abort_flag = flags + kFlagAbort;
  const uint32_t smem_base = smem_addr(smem);
  unsigned char* ring = smem + (((smem_base + SH::FIXED + 1023u) & ~1023u) - smem_base);
  unsigned char* qslot = ring + static_cast<size_t>(NST) * STAGE;  // [2][HG][G][D] fp16
  int* pfx = reinterpret_cast<int*>(qslot + 2 * QSLOT);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.num_seqs;
  const int Hkv = p.num_kv_heads;
  const int NHG = Hkv / HG;
  const int cap = (p.max_blocks - (PFX ? p.pfx_blocks : 0)) * BS;
  const int loff = PFX ? p.pfx_blocks * BS : 0;  // tokens before the streamed part

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), HG);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(smem_addr(&qfull_bar[q]), 1);
      mbar_init(smem_addr(&qempty_bar[q]), HG);
    }
    for (int m = 0; m < kMsgSlots; ++m) {
      mbar_init(smem_addr(&mfull_bar[m]), HG);  // one arrival per consumer warp
      mbar_init(smem_addr(&mempty_bar[m]), kMergeWarps);
    }
    flags[kFlagAbort] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  if constexpr (!PFX) {
    // Every input may still be written by the kernel launched just before
    // this one on the stream (programmatic dependent launch), so none is read
    // before griddepcontrol.wait. The CTAs only ask L2 for the lengths, the
    // block table and q meanwhile, spread over the grid (L2 stays coherent
    // with whatever that kernel writes, so a prefetch is never stale).
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long me = static_cast<long long>(blockIdx.x) * blockDim.x + tid;
    const long long len_lines = (static_cast<long long>(S) * 4 + 127) / 128;
    const long long tab_lines = (static_cast<long long>(S) * p.max_blocks * 4 + 127) / 128;
    const long long q_lines = (static_cast<long long>(S) * p.num_q_heads * D * 2 + 127) / 128;
    const long long n_lines = len_lines + min(tab_lines + q_lines, kPrefetchLines);
    for (long long i = me; i < n_lines; i += nthreads) {
      const char* a;
      if (i < len_lines)
        a = reinterpret_cast<const char*>(p.seq_lens) + i * 128;
      else if (i < len_lines + tab_lines)
        a = reinterpret_cast<const char*>(p.block_table) + (i - len_lines) * 128;
      else
        a = reinterpret_cast<const char*>(p.q) + (i - len_lines - tab_lines) * 128;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }

  // ---- blocks per sequence, exclusive prefix sum in shared memory ----
  block_prefix(pfx, flags + kFlagWsum, p.seq_lens, S, BS, cap, p.err, loff);
  const Geometry geo = chunk_geometry(pfx[S] * NHG, gridDim.x, p.cap_blocks);
  const int chunk = geo.chunk;
  const bool has_work = static_cast<int>(blockIdx.x) < geo.nchunks;

  // The producer's first two pieces, and an L2 prefetch of their table
  // entries and q rows.
  Walk wk;
  Piece P{}, PN{};
  bool have = false, nhave = false;
  int lraw_first = 0;  // the first piece's sequence length, as given
  if (warp == HG) {
    walk_begin(wk, blockIdx.x, geo, pfx, S, NHG);
    have = walk_next(wk, geo, gridDim.x, pfx, S, NHG, P);
    if (have) lraw_first = __ldg(p.seq_lens + P.cur.seq);
    nhave = have && walk_next(wk, geo, gridDim.x, pfx, S, NHG, PN);
    for (int k = 0; k < 2; ++k) {
      const Piece& X = k == 0 ? P : PN;
      if (!(k == 0 ? have : nhave)) break;
      const int32_t* trow =
          p.block_table + static_cast<long long>(X.cur.seq) * p.max_blocks + X.cur.j;
      if (lane < min(32, X.n)) asm volatile("prefetch.global.L2 [%0];" ::"l"(trow + lane));
      const char* qrow = reinterpret_cast<const char*>(
          p.q + (static_cast<long long>(X.cur.seq) * p.num_q_heads +
                 static_cast<long long>(X.cur.hg) * HG * G) * D);
      for (int off = lane * 128; off < QSLOT; off += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + off));
    }
  }

  // In shared-prefix mode the kernel launched just before this one is the
  // prefix kernel, which writes only the prefix records and lets this kernel
  // start once everything launched before it has completed: the lengths,
  // table, q and pools may be read at once, and the wait sits before the
  // first read of a prefix record (pfx_wait), so the streaming overlaps the
  // prefix kernel.
  // A dependent kernel launched after this one may start its own prologue.
  asm volatile("griddepcontrol.launch_dependents;");

  if (warp == HG) {
    // =========================== producer warp ===========================
    // Streams the CTA's pieces, each in groups of up to 32 blocks. For each
    // piece it first publishes, in q slot (piece & 1), the piece's metadata
    // and its HG*G q rows. The table entries (and length) of the next group,
    // in this piece or the next, are loaded while the current group is issued
    // and used only once it is: no group or piece boundary waits on a global
    // load, and no load holds up the current group's copies.
    uint32_t g = 0;   // ring sequence number (stages)
    uint32_t pc = 0;  // piece number
    const uint64_t stream_pol = KV8 ? 0ull : l2_evict_first_policy();
    // stages and q slots whose copies were issued (after an abort the walk
    // goes on without issuing, so g and pc run ahead of these)
    uint32_t g_iss = 0, pc_iss = 0;
    int j0 = 0;
    int phys_cur = 0, len_cur = 0;
    // append mode: the current piece's appended row (its head group's part)
    // when the piece holds its segment's last block a_blk
    constexpr int kAV = (kMaxHG * D / 8 + 31) / 32;  // 16-byte vectors per lane
    uint4 ak[kAV], av[kAV];
    int a_blk = -1, a_slot = -1;
    if (have) {
      len_cur = min(max(lraw_first - loff, 0), cap);
      phys_cur = lane < min(32, P.n)
                     ? __ldg(p.block_table + static_cast<long long>(P.cur.seq) * p.max_blocks +
                             P.cur.j + lane)
                     : 0;
    }
    while (have) {
      if (j0 == 0) {
        // new piece: metadata and q rows -> q slot (pc & 1)
        const int qs = static_cast<int>(pc & 1);
        if (!__shfl_sync(0xffffffffu, *abort_flag, 0) &&
            (pc < 2 ||
             warp_wait_phase(smem_addr(&qempty_bar[qs]), ((pc >> 1) - 1) & 1, abort_flag, p.err, p.wait_ns))) {
          if (lane == 0) {
            PieceMeta* m = pmeta + qs;
            m->seq = P.cur.seq;
            m->hg = P.cur.hg;
            m->j = P.cur.j;
            m->n = P.n;
            m->nb = P.cur.nb;
            m->len = len_cur;
            m->s0 = P.cur.seg_start;
            m->c = P.c;
            m->last = nhave ? 0 : 1;
            const uint32_t qb = smem_addr(&qfull_bar[qs]);
            // the arrival releases the metadata stores above
            mbar_arrive_expect_tx(qb, QSLOT);
            bulk_copy_g2s(smem_addr(qslot + qs * QSLOT),
                          p.q + (static_cast<long long>(P.cur.seq) * p.num_q_heads +
                                 static_cast<long long>(P.cur.hg) * HG * G) * D,
                          QSLOT, qb);
          }
          pc_iss = pc + 1;
          __syncwarp();
        }
        if constexpr (!KV8 && !PFX) {
          // append mode: the new row of the piece's sequence is loaded now,
          // used when its block's copy is issued
          a_blk = -1;
          if (p.k_new != nullptr && len_cur > 0) {
            const int lb = (len_cur - 1) / BS;
            if (lb >= P.cur.j && lb < P.cur.j + P.n) {
              a_blk = lb;
              a_slot = __ldg(p.slot_mapping + P.cur.seq);
              const long long src =
                  (static_cast<long long>(P.cur.seq) * p.num_kv_heads + P.cur.hg * HG) * (D / 8);
              const uint4* kn = reinterpret_cast<const uint4*>(p.k_new) + src;
              const uint4* vn = reinterpret_cast<const uint4*>(p.v_new) + src;
#pragma unroll
              for (int i = 0; i < kAV; ++i) {
                const int idx = lane + 32 * i;
                if (idx < HG * D / 8) {
                  ak[i] = __ldg(kn + idx);
                  av[i] = __ldg(vn + idx);
                }
              }
            }
          }
        }
      }
      const int nn = min(32, P.n - j0);
      // table entries (and raw length) of the next group
      const bool next_in_piece = j0 + 32 < P.n;
      int phys_nxt = 0, lraw_nxt = 0;
      if (next_in_piece) {
        if (lane < min(32, P.n - j0 - 32))
          phys_nxt = __ldg(p.block_table + static_cast<long long>(P.cur.seq) * p.max_blocks +
                           P.cur.j + j0 + 32 + lane);
      } else if (nhave) {
        lraw_nxt = __ldg(p.seq_lens + PN.cur.seq);
        if (lane < min(32, PN.n))
          phys_nxt = __ldg(p.block_table + static_cast<long long>(PN.cur.seq) * p.max_blocks +
                           PN.cur.j + lane);
      }
      for (int jj = 0; jj < nn; ++jj) {
        const int phys = __shfl_sync(0xffffffffu, phys_cur, jj);
        const int blk = P.cur.j + j0 + jj;
        const int vb = min(BS, len_cur - blk * BS);  // valid rows of the block (>= 1)
        const int nsb = (vb + TS - 1) / TS;           // stages that hold valid rows
        const bool bad = phys < 0 || phys >= p.num_blocks;
        if constexpr (!KV8 && !PFX) {
          if (blk == a_blk) {
            // append mode: the sequence's new row (its last token) is written
            // into this block before any of its copies is issued; a slot
            // that is not that row is refused
            const int row = (len_cur - 1) % BS;
            const bool ok_slot = !bad && a_slot == phys * BS + row;
            if (a_slot >= 0 && !ok_slot && lane == 0) atomicOr(p.err, PA_DEVERR_BAD_SLOT);
            if (ok_slot) {
              const long long off =
                  static_cast<long long>(phys) * p.block_stride +
                  (static_cast<long long>(row) * p.num_kv_heads + P.cur.hg * HG) * D;
              uint4* kd = reinterpret_cast<uint4*>(const_cast<__half*>(p.k_pool) + off);
              uint4* vd = reinterpret_cast<uint4*>(const_cast<__half*>(p.v_pool) + off);
#pragma unroll
              for (int i = 0; i < kAV; ++i) {
                const int idx = lane + 32 * i;
                if (idx < HG * D / 8) {
                  kd[idx] = ak[i];
                  vd[idx] = av[i];
                }
              }
              // the block's copies (async proxy) read what was just written
              asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            __syncwarp();
          }
        }
        for (int sb = 0; sb < nsb; ++sb, ++g) {
          const int stage = g % NST;
          const uint32_t use = g / NST;
          if (__shfl_sync(0xffffffffu, *abort_flag, 0)) continue;
          if (use > 0 &&
              !warp_wait_phase(smem_addr(&empty_bar[stage]), (use - 1) & 1, abort_flag, p.err, p.wait_ns))
            continue;
          if (lane == 0) {
            const uint32_t fb = smem_addr(&full_bar[stage]);
            if (bad) atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
            // whole tiles: rows past the sequence end are masked by the consumers
            mbar_arrive_expect_tx(fb, bad ? 0u : static_cast<uint32_t>(STAGE));
            if (!bad) {
              const uint32_t kdst = smem_addr(ring + static_cast<size_t>(stage) * STAGE);
#pragma unroll
              for (int h = 0; h < SH::NHALF; ++h) {
                const int x = (128 / SH::ESZ) * h;  // first value of the 128-byte line
                if constexpr (KV8) {
                  tma_load_4d(kdst + h * HALF, &kmap, x, sb * TS, P.cur.hg * HG, phys, fb);
                  tma_load_4d(kdst + TILE + h * HALF, &vmap, x, sb * TS, P.cur.hg * HG, phys, fb);
                } else {
                  tma_load_4d_once(kdst + h * HALF, &kmap, x, sb * TS, P.cur.hg * HG, phys, fb,
                                   stream_pol);
                  tma_load_4d_once(kdst + TILE + h * HALF, &vmap, x, sb * TS, P.cur.hg * HG, phys,
                                   fb, stream_pol);
                }
              }
            }
          }
          g_iss = g + 1;
          __syncwarp();
        }
      }
      if (next_in_piece) {
        j0 += 32;
      } else {
        ++pc;
        P = PN;
        have = nhave;
        j0 = 0;
        len_cur = min(max(lraw_nxt - loff, 0), cap);
        if (have) nhave = walk_next(wk, geo, gridDim.x, pfx, S, NHG, PN);
      }
      phys_cur = phys_nxt;
    }
    // After an abort, wait (bounded, on the full limit whatever the pipeline
    // waits used) for copies still landing in shared memory: the last NST
    // stages and the last two q slots issued. Each of those barriers has one
    // phase pending, the one waited for; every earlier phase of its slot
    // completed before the slot was issued again.
    if (*abort_flag) {
      const uint32_t first = g_iss > static_cast<uint32_t>(NST) ? g_iss - NST : 0;
      for (uint32_t gi = first; gi < g_iss; ++gi) {
        const uint32_t bar = smem_addr(&full_bar[gi % NST]);
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(bar, (gi / NST) & 1) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
      for (uint32_t pi = pc_iss > 2 ? pc_iss - 2 : 0; pi < pc_iss; ++pi) {
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(smem_addr(&qfull_bar[pi & 1]), (pi >> 1) & 1) &&
               global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    return;
  }

  if (warp > HG) {
    // ============================= merge warps ============================
    // For every cut piece that is not the CTA's last, the consumer warps send
    // a message (slot m % kMsgSlots) once all their records are written. Each
    // merge warp counts one arrival for each of its heads (head h belongs to
    // merge warp h % kMergeWarps, lane h counts it) and merges each of its
    // heads whose arrivals are complete. A stop message ends the loop.
    const int mw = warp - HG - 1;
    for (uint32_t mc = 0; has_work; ++mc) {
      const int ms = static_cast<int>(mc % kMsgSlots);
      if (!warp_wait_phase<256>(smem_addr(&mfull_bar[ms]), (mc / kMsgSlots) & 1, abort_flag,
                                p.err, p.wait_ns))
        break;
      const MsgMeta msg = mmeta[ms];
      // the consumers' records (ordered before their arrivals on the barrier)
      // become visible to the whole GPU before any arrival is counted
      fence_acq_rel_gpu();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&mempty_bar[ms]));
      if (msg.stop) break;
      const int s0 = msg.s0;
      const int c_first = s0 / chunk, c_last = (s0 + msg.nb - 1) / chunk;
      const int E = c_last - c_first + 1;
      unsigned long long* words =
          p.counters + static_cast<long long>(msg.seq) * Hkv + static_cast<long long>(msg.hg) * HG;
      const bool mine = lane < HG && lane % kMergeWarps == mw;
      const bool done =
          mine && arrive_last(words + lane, p.tag, static_cast<unsigned>(E), 0ull, p.err);
      unsigned last = __ballot_sync(0xffffffffu, done);
      if (last) fence_acq_rel_gpu();  // acquire: the other chunks' records are visible
      while (last) {
        const int h = __ffs(last) - 1;
        last &= last - 1;
        const int kvh_m = msg.hg * HG + h;
        auto rec_of = [&](int i) -> long long {
          if (PFX && i >= E)
            return p.pfx_rec_base +
                   (static_cast<long long>(i - E) * S + msg.seq) * Hkv + kvh_m;
          return record_index(c_first + i, c_first, s0, chunk, HG, h);
        };
        __half* out_row = p.out + (static_cast<long long>(msg.seq) * p.num_q_heads +
                                   static_cast<long long>(kvh_m) * G) * D;
        pfx_wait<PFX>();
        merge_partials<D, G>(p.records, E + (PFX ? p.pfx_chunks : 0), rec_of, out_row);
      }
    }
    return;
  }

  // ============================ consumer warps ============================
  // Warp w owns KV head (group * HG + w) and its G query heads.
  const int w = warp;
  const int gid = lane >> 2;  // mma group id: row of A / column of B
  const int tig = lane & 3;   // thread in group

  // outputs of sequences with nothing to stream (this CTA's share): zero, or
  // in shared-prefix mode the merge of the prefix records alone
  for (int i = blockIdx.x; i < S; i += gridDim.x) {
    if (pfx[i + 1] == pfx[i]) {
      if constexpr (PFX) {
        pfx_wait<PFX>();
        for (int kv = w; kv < Hkv; kv += HG) {
          auto rec_of = [&](int k) -> long long {
            return p.pfx_rec_base + (static_cast<long long>(k) * S + i) * Hkv + kv;
          };
          merge_partials<D, G>(p.records, p.pfx_chunks, rec_of,
                               p.out + (static_cast<long long>(i) * p.num_q_heads +
                                        static_cast<long long>(kv) * G) * D);
        }
      } else {
        __half* o = p.out + static_cast<long long>(i) * p.num_q_heads * D;
        for (int e = tid; e < p.num_q_heads * D; e += HG * 32) o[e] = __float2half_rn(0.f);
      }
    }
  }
  if (!has_work) return;

  // ldmatrix addressing inside a swizzled tile: lane supplies row (lane & 7)
  // of matrix (lane >> 3); logical 16-byte chunk c of row r sits at chunk
  // c ^ (r & 7) of its 128-byte line. A head's rows start at a multiple of 8
  // rows, so r & 7 == lane & 7 for every row a lane addresses.
  const int ld_row = lane & 7;
  const int ld_mat = lane >> 3;

  uint32_t g = 0;   // ring sequence number of the next stage
  uint32_t mc = 0;  // messages sent to the merge warps
  for (uint32_t pc = 0;; ++pc) {
    // ---- the piece: metadata and q from q slot (pc & 1) ----
    const int qs = static_cast<int>(pc & 1);
    const bool qok = warp_wait_phase(smem_addr(&qfull_bar[qs]), (pc >> 1) & 1, abort_flag, p.err, p.wait_ns);
    if (!qok) break;
    const PieceMeta pm = pmeta[qs];
    const int pj = pm.j, n = pm.n, L = pm.len;
    const int kvh = pm.hg * HG + w;
    // in shared-prefix mode every piece is merged with the prefix records
    const bool cut = PFX || pj > 0 || pj + n < pm.nb;
    __half* out_row = p.out + (static_cast<long long>(pm.seq) * p.num_q_heads +
                               static_cast<long long>(kvh) * G) * D;
    // a cut piece's partial record: slot 0 if the piece starts its chunk, else 1
    // (in shared-prefix mode a whole segment uses its (sequence, KV head) slot)
    const int s0 = pm.s0;
    const bool whole = !(pj > 0 || pj + n < pm.nb);
    float* rec = p.records +
                 (PFX && whole
                      ? p.pfx_own_base + static_cast<long long>(pm.seq) * Hkv + kvh
                      : (2ll * pm.c + (s0 + pj == pm.c * chunk ? 0 : 1)) * HG + w) *
                     static_cast<long long>(SH::REC);
    if constexpr (KV8) {
      // ---- fp8 pools: E4M3 tiles, converted to fp16 fragments in registers ----
      // Scores as S^T = K Q^T: the 16 tokens of a stage are the M rows, the
      // heads the N columns, so a stage takes D/16 mma. The K fragments come
      // from ldmatrix on byte pairs: lane (gid, tig) gets 4 consecutive values
      // (dims 4*tig .. +3 of a 16-dim chunk) of token gid (and gid + 8); the
      // dot product's order over dims is free, so mma k-index 2*tig + e takes
      // dim 4*tig + e and k-index 2*tig + 8 + e takes dim 4*tig + 2 + e, and q
      // is loaded in the same order. k_scale folds into the score scale and
      // v_scale into the result.
      uint32_t qb[D / 16][2];
      {
        const unsigned char* qrow =
            qslot + qs * QSLOT + (w * G + (gid < G ? gid : 0)) * (D * 2);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          const uint2 v = *reinterpret_cast<const uint2*>(qrow + (16 * c + 4 * tig) * 2);
          qb[c][0] = gid < G ? v.x : 0u;
          qb[c][1] = gid < G ? v.y : 0u;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&qempty_bar[qs]));
      }
      const float qsc = p.qscale * __ldg(p.k_scale + kvh);
      const float vsc = __ldg(p.v_scale + kvh);
      float m0 = -INFINITY, m1 = -INFINITY;  // heads 2*tig, 2*tig+1: running max (log2 units)
      float l0 = 0.f, l1 = 0.f;              // and partial sums over this lane's tokens
      float o[D / 16][4];                    // O^T[dim 16*mt + 2*gid (+1)][head 2*tig (+1)]
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      const int tok = ((ld_mat & 1) << 3) + ld_row;  // row this lane addresses for ldmatrix

      for (int jj = 0; jj < n; ++jj) {
        const int blk = pj + jj;
        const int vb = min(BS, L - blk * BS);
        const int nsb = (vb + TS - 1) / TS;
        for (int sb = 0; sb < nsb; ++sb, ++g) {
          const int stage = g % NST;
          if (!warp_wait_phase(smem_addr(&full_bar[stage]), (g / NST) & 1, abort_flag, p.err, p.wait_ns))
            continue;
          const int rows = min(TS, vb - sb * TS);
          unsigned char* kt = ring + static_cast<size_t>(stage) * STAGE;
          unsigned char* vt = kt + TILE;
          if (rows < TS) {
            // rows past the sequence end must add exactly zero to P V
            uint4* z = reinterpret_cast<uint4*>(vt + (w * TS + rows) * 128);
            for (int i = lane; i < (TS - rows) * 8; i += 32) z[i] = make_uint4(0, 0, 0, 0);
            __syncwarp();
          }
          const uint32_t kaddr = smem_addr(kt) + w * TS * 128;
          const uint32_t vaddr = smem_addr(vt) + w * TS * 128;

          // ---- S^T = K Q^T ----
          float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            // matrices: tokens 0-7 / 8-15 of 16-dim chunks 2*cc and 2*cc + 1
            const int ch = 2 * cc + (ld_mat >> 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kaddr + tok * 128 + ((ch ^ ld_row) << 4), r0, r1, r2, r3);
            mma_16816(sc, e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                      e4m3x2_to_f16x2(r1 >> 16), qb[2 * cc][0], qb[2 * cc][1]);
            mma_16816(sc, e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                      e4m3x2_to_f16x2(r3 >> 16), qb[2 * cc + 1][0], qb[2 * cc + 1][1]);
          }
          // ---- online softmax per head over the stage's tokens ----
          // sc: [token gid][head 2tig], [gid][2tig+1], [gid+8][2tig], [gid+8][2tig+1]
          const bool t0 = gid < rows, t1 = gid + 8 < rows;
          const float x0 = t0 ? sc[0] * qsc : -INFINITY;
          const float x1 = t0 ? sc[1] * qsc : -INFINITY;
          const float x2 = t1 ? sc[2] * qsc : -INFINITY;
          const float x3 = t1 ? sc[3] * qsc : -INFINITY;
          float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
          const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = fast_exp2(m0 - mu0), al1 = fast_exp2(m1 - mu1);
          m0 = mn0;
          m1 = mn1;
          const float p0 = fast_exp2(x0 - mu0), p1 = fast_exp2(x1 - mu1);
          const float p2 = fast_exp2(x2 - mu0), p3 = fast_exp2(x3 - mu1);
          l0 = l0 * al0 + p0 + p2;
          l1 = l1 * al1 + p1 + p3;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
          }
          // P^T as the B operand (k = token, n = head): transpose the two
          // 8x8 blocks (tokens 0-7 and 8-15) of P held [token][head]
          const uint32_t pb0 = movmatrix_trans(pack_half2(p0, p1));
          const uint32_t pb1 = movmatrix_trans(pack_half2(p2, p3));
          // ---- O^T += V^T P^T ----
          // ldmatrix.trans on byte pairs gives lane (gid, tig) the bytes
          // V[2tig][d], V[2tig][d+1], V[2tig+1][d], V[2tig+1][d+1] with
          // d = 2*gid of the chunk; A row gid takes dim d and row gid + 8 dim
          // d + 1 (the rows of O^T are then those dims).
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            const int ch = 2 * cc + (ld_mat >> 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(vaddr + tok * 128 + ((ch ^ ld_row) << 4), r0, r1, r2, r3);
            const uint32_t u0 = prmt(r0, 0u, 0x3120u), u1 = prmt(r1, 0u, 0x3120u);
            const uint32_t u2 = prmt(r2, 0u, 0x3120u), u3 = prmt(r3, 0u, 0x3120u);
            mma_16816(o[2 * cc], e4m3x2_to_f16x2(u0), e4m3x2_to_f16x2(u0 >> 16),
                      e4m3x2_to_f16x2(u1), e4m3x2_to_f16x2(u1 >> 16), pb0, pb1);
            mma_16816(o[2 * cc + 1], e4m3x2_to_f16x2(u2), e4m3x2_to_f16x2(u2 >> 16),
                      e4m3x2_to_f16x2(u3), e4m3x2_to_f16x2(u3 >> 16), pb0, pb1);
          }
          if (rows < TS) fence_proxy_async_smem();  // generic zero-fill before the next TMA write
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
        }
      }

      // ---- piece finished: sums over all tokens of the piece ----
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      const int h0 = 2 * tig, h1 = 2 * tig + 1;
      if (!cut) {
        const float i0 = l0 > 0.f ? vsc / l0 : 0.f, i1 = l1 > 0.f ? vsc / l1 : 0.f;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d = mt * 16 + 2 * gid;
          if (h0 < G)
            *reinterpret_cast<__half2*>(out_row + h0 * D + d) =
                __floats2half2_rn(o[mt][0] * i0, o[mt][2] * i0);
          if (h1 < G)
            *reinterpret_cast<__half2*>(out_row + h1 * D + d) =
                __floats2half2_rn(o[mt][1] * i1, o[mt][3] * i1);
        }
      } else {
        // the record holds the dequantized accumulator (v_scale applied)
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d = mt * 16 + 2 * gid;
          if (h0 < G)
            *reinterpret_cast<float2*>(rec + h0 * D + d) = make_float2(o[mt][0] * vsc, o[mt][2] * vsc);
          if (h1 < G)
            *reinterpret_cast<float2*>(rec + h1 * D + d) = make_float2(o[mt][1] * vsc, o[mt][3] * vsc);
        }
        if (gid == 0) {
          if (h0 < G) {
            rec[G * D + 2 * h0] = m0;
            rec[G * D + 2 * h0 + 1] = l0;
          }
          if (h1 < G) {
            rec[G * D + 2 * h1] = m1;
            rec[G * D + 2 * h1 + 1] = l1;
          }
        }
      }
    } else {
      // fp16 consumer tiling
      constexpr int KSTEPS = D / 16;  // QK k-steps over head_dim
      constexpr int MT = D / 16;      // PV m-tiles over head_dim
      constexpr int NT = TS / 8;      // 8-token groups per stage
      constexpr int PK = (NT + 1) / 2;  // PV k-steps (16 tokens) per stage
      uint32_t qa[KSTEPS][2];  // A fragments a0/a2 per k-step; rows (heads) >= G are zero
      {
        const uint32_t qrow = smem_addr(qslot + qs * QSLOT) +
                              (w * G + (ld_row < G ? ld_row : 0)) * (D * 2);
  #pragma unroll
        for (int kk = 0; kk < KSTEPS; kk += 2) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(qrow + (2 * kk + ld_mat) * 16, r0, r1, r2, r3);
          qa[kk][0] = gid < G ? r0 : 0u;
          qa[kk][1] = gid < G ? r1 : 0u;
          qa[kk + 1][0] = gid < G ? r2 : 0u;
          qa[kk + 1][1] = gid < G ? r3 : 0u;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&qempty_bar[qs]));
      }

        float m_run = -INFINITY, l_run = 0.f;  // head gid: running max (log2 units), partial sum
        float o[MT][4];                     // O^T[d = mt*16 + gid (+8)][h = 2*tig (+1)]
  #pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

        for (int jj = 0; jj < n; ++jj) {
          const int blk = pj + jj;
          const int vb = min(BS, L - blk * BS);
          const int nsb = (vb + TS - 1) / TS;
          for (int sb = 0; sb < nsb; ++sb, ++g) {
            const int stage = g % NST;
            if (!warp_wait_phase(smem_addr(&full_bar[stage]), (g / NST) & 1, abort_flag, p.err, p.wait_ns))
              continue;
            const int rows = min(TS, vb - sb * TS);
            unsigned char* kt = ring + static_cast<size_t>(stage) * STAGE;
            unsigned char* vt = kt + TILE;
            if (rows < TS) {
              // rows past the sequence end must add exactly zero to P V
              const int words = (TS - rows) * 8;  // 16-byte words per half
  #pragma unroll
              for (int h = 0; h < SH::NHALF; ++h) {
                uint4* z = reinterpret_cast<uint4*>(vt + h * HALF + (w * TS + rows) * 128);
                for (int i = lane; i < words; i += 32) z[i] = make_uint4(0, 0, 0, 0);
              }
              __syncwarp();
            }
            const uint32_t kaddr = smem_addr(kt) + w * TS * 128;
            const uint32_t vaddr = smem_addr(vt) + w * TS * 128;

            // ---- S = Q K^T for each 8-token group ----
            // x4 of k-steps (kk, kk+1): matrix m covers dims (2*kk + m) * 8 .. +8
            float s[NT][4];
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
              const uint32_t rowa = kaddr + (nt * 8 + ld_row) * 128;
  #pragma unroll
              for (int kk = 0; kk < KSTEPS; kk += 2) {
                const int gc = 2 * kk + ld_mat;  // 16-byte chunk of the row, 0 .. D/8-1
                uint32_t b0, b1, b2, b3;
                ldsm_x4(rowa + (gc >> 3) * HALF + (((gc & 7) ^ ld_row) << 4), b0, b1, b2, b3);
                mma_16816(s[nt], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                mma_16816(s[nt], qa[kk + 1][0], 0u, qa[kk + 1][1], 0u, b2, b3);
              }
            }
            // ---- online softmax over this stage's tokens (row gid = head) ----
            float mx = -INFINITY;
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
  #pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int t = nt * 8 + 2 * tig + e;
                const float v = t < rows ? s[nt][e] * p.qscale : -INFINITY;
                s[nt][e] = v;
                mx = fmaxf(mx, v);
              }
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float mu = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = fast_exp2(m_run - mu);
            m_run = m_new;
            float ps = 0.f;
            uint32_t pb[NT];  // P as fp16 pairs: B operand of the PV mma
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float p0 = fast_exp2(s[nt][0] - mu);
              const float p1 = fast_exp2(s[nt][1] - mu);
              ps += p0 + p1;
              pb[nt] = pack_half2(p0, p1);
            }
            l_run = l_run * alpha + ps;
            // rescale O^T columns: heads 2*tig and 2*tig+1 live in mma groups 2*tig, 2*tig+1
            const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * tig);
            const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * tig + 4);
  #pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              o[mt][0] *= a_lo;
              o[mt][1] *= a_hi;
              o[mt][2] *= a_lo;
              o[mt][3] *= a_hi;
            }
            // ---- O^T += V^T P^T over 16-token k-steps ----
            // x4.trans of m-tile mt: matrix m covers tokens +8*(m>>1), dims mt*16 + 8*(m&1)
  #pragma unroll
            for (int pk = 0; pk < PK; ++pk) {
              const uint32_t pb0 = pb[2 * pk];
              const uint32_t pb1 = (2 * pk + 1 < NT) ? pb[2 * pk + 1] : 0u;
              const uint32_t rowa = vaddr + (pk * 16 + ld_row + (ld_mat >> 1) * 8) * 128;
  #pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                const int gc = 2 * mt + (ld_mat & 1);
                const uint32_t addr = rowa + (gc >> 3) * HALF + (((gc & 7) ^ ld_row) << 4);
                uint32_t a0, a1, a2, a3;
                if (2 * pk + 1 < NT) {
                  ldsm_x4_t(addr, a0, a1, a2, a3);
                } else {
                  ldsm_x2_t(addr, a0, a1);
                  a2 = a3 = 0u;
                }
                mma_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
              }
            }
            if (rows < TS) fence_proxy_async_smem();  // generic zero-fill before the next TMA write
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
          }
        }

        // ---- piece finished: this warp holds its head's whole state ----
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
        const int h0 = 2 * tig, h1 = 2 * tig + 1;
        if (!cut) {
          const float l0 = __shfl_sync(0xffffffffu, l_run, 8 * tig);
          const float l1 = __shfl_sync(0xffffffffu, l_run, 8 * tig + 4);
          const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
  #pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int d = mt * 16 + gid;
            if (h0 < G) {
              out_row[h0 * D + d] = __float2half_rn(o[mt][0] * i0);
              out_row[h0 * D + d + 8] = __float2half_rn(o[mt][2] * i0);
            }
            if (h1 < G) {
              out_row[h1 * D + d] = __float2half_rn(o[mt][1] * i1);
              out_row[h1 * D + d + 8] = __float2half_rn(o[mt][3] * i1);
            }
          }
        } else {
          // cut segment: this chunk's partial record
  #pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int d = mt * 16 + gid;
            if (h0 < G) {
              rec[h0 * D + d] = o[mt][0];
              rec[h0 * D + d + 8] = o[mt][2];
            }
            if (h1 < G) {
              rec[h1 * D + d] = o[mt][1];
              rec[h1 * D + d + 8] = o[mt][3];
            }
          }
          if (tig == 0 && gid < G) {
            rec[G * D + 2 * gid] = m_run;
            rec[G * D + 2 * gid + 1] = l_run;
          }
        }
    }
    if (PFX && whole) {
      // the whole segment is here: merge it with the prefix records now
      __syncwarp();  // the record's lanes, before any lane reads it back
      auto rec_of = [&](int i) -> long long {
        if (i == 0) return p.pfx_own_base + static_cast<long long>(pm.seq) * Hkv + kvh;
        return p.pfx_rec_base + (static_cast<long long>(i - 1) * S + pm.seq) * Hkv + kvh;
      };
      pfx_wait<PFX>();
      merge_partials<D, G>(p.records, 1 + p.pfx_chunks, rec_of, out_row);
    } else if (cut) {
          if (!pm.last) {
            // hand the arrival (and any merge) to the merge warps: the warp
            // barrier orders every lane's record stores before lane 0's arrival,
            // whose release makes them visible to the merge warps' acquire
            if (mc >= kMsgSlots)
              warp_wait_phase(smem_addr(&mempty_bar[mc % kMsgSlots]), ((mc / kMsgSlots) - 1) & 1,
                              abort_flag, p.err, p.wait_ns);
            if (w == 0 && lane == 0) {
              MsgMeta* m = mmeta + mc % kMsgSlots;
              m->seq = pm.seq;
              m->hg = pm.hg;
              m->nb = pm.nb;
              m->s0 = s0;
              m->stop = 0;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&mfull_bar[mc % kMsgSlots]));
            ++mc;
          } else {
            // The CTA's last piece: count the arrival here and merge if it
            // completes the segment, which it usually does (the other chunks'
            // pieces are mostly done). First try to claim the last arrival
            // outright: a last arrival's record is read by no other warp, so it
            // needs no release and the claim does not wait for its stores.
            // Otherwise release the record and count the arrival as usual.
            __syncwarp();  // the record's lanes, before any lane reads it back
            const int c_first = s0 / chunk, c_last = (s0 + pm.nb - 1) / chunk;
            const int E = c_last - c_first + 1;
            unsigned long long* word = p.counters + static_cast<long long>(pm.seq) * Hkv + kvh;
            const unsigned long long claim = (p.tag << kArrivalBits) | static_cast<unsigned>(E - 1);
            int done = 0;
            unsigned long long seen = 0;
            if (lane == 0) {
              seen = atomicCAS(word, claim, 0ull);
              done = seen == claim;
            }
            done = __shfl_sync(0xffffffffu, done, 0);
            if (!done) {
              fence_acq_rel_gpu();  // release: the record is visible before the arrival
              __syncwarp();
              // the failed claim returned the word: the arrival starts from it
              if (lane == 0) done = arrive_last(word, p.tag, static_cast<unsigned>(E), seen, p.err);
              done = __shfl_sync(0xffffffffu, done, 0);
            }
            if (done) {
              // acquire: the other chunks' records are visible to this warp
              fence_acq_rel_gpu();
              auto rec_of = [&](int i) -> long long {
                if (PFX && i >= E)
                  return p.pfx_rec_base +
                         (static_cast<long long>(i - E) * S + pm.seq) * Hkv + kvh;
                return record_index(c_first + i, c_first, s0, chunk, HG, w);
              };
              pfx_wait<PFX>();
              merge_partials<D, G>(p.records, E + (PFX ? p.pfx_chunks : 0), rec_of, out_row);
            }
          }
    }
    if (pm.last) break;
  }
  // tell the merge warps there is nothing more
  if (!*abort_flag) {
    if (mc >= kMsgSlots)
      warp_wait_phase(smem_addr(&mempty_bar[mc % kMsgSlots]), ((mc / kMsgSlots) - 1) & 1,
                      abort_flag, p.err, p.wait_ns);
    if (w == 0 && lane == 0) mmeta[mc % kMsgSlots].stop = 1;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&mfull_bar[mc % kMsgSlots]));
  }
}


// --------------------------------------------------------------- host ---
size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Chunks a launch can produce: at most one per CTA of the grid (kMaxGrid),
// or, with a per-chunk cap, enough to cover every block of every segment.
long long max_chunks(int S, int nhg, int MB, int cap_blocks) {
  long long m = kMaxGrid;
  if (cap_blocks > 0) {
    const long long blocks = static_cast<long long>(S) * nhg * MB;
    const long long need = (blocks + cap_blocks - 1) / cap_blocks;
    if (need > m) m = need;
  }
  return m;
}

struct Layout {
  size_t counters = 0, records = 0, total = 0;
};

// Workspace: arrival counters (8 bytes per sequence and KV head), then two
// partial records per chunk and KV head of the group (written by CTAs whose
// chunk cuts a segment, read by the warp that merges it). No part of it needs
// initialising: counter words carry the tag of the call that wrote them.
Layout workspace_layout(int S, int Hq, int Hkv, int D, int MB, int cap_blocks) {
  Layout w;
  const int G = Hq / Hkv;
  const int hg = head_group(Hkv);
  const long long recs = 2 * max_chunks(S, Hkv / hg, MB, cap_blocks) * hg;
  w.counters = 0;
  w.records = round256(static_cast<size_t>(S) * Hkv * 8);
  w.total = w.records + round256(static_cast<size_t>(recs) * rec_floats(G, D) * 4);
  return w;
}

// Time limit of the attention kernel's pipeline waits (pa_set_wait_limit_ns).
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};

// Tag of the next decode call: unique within the process (2^44 values), never
// zero, so a zero counter word always reads as "no arrivals".
unsigned long long next_call_tag() {
  static std::atomic<unsigned long long> counter{0};
  constexpr unsigned long long kTagMask = (1ull << (64 - kArrivalBits)) - 1;
  unsigned long long t = (counter.fetch_add(1, std::memory_order_relaxed) + 1) & kTagMask;
  return t == 0 ? 1 : t;
}

// Launch shape of one decode: head group, ring depth, threads, shared memory
// and the persistent grid (SMs x resident CTAs, at most kMaxGrid).
struct LaunchCfg {
  int hg = 0, nst = 0, threads = 0;
  size_t smem = 0;
  long long grid = 0;
};

template <int D, int BS, int G, bool KV8 = false, bool PFX = false>
pa_status launch_config(const pa::DeviceInfo& dev, int S, int Hkv, LaunchCfg* cfg) {
  using SH = Shape<D, BS, G, KV8>;
  auto kernel = paged_decode_kernel<D, BS, G, KV8, PFX>;
  cfg->hg = head_group(Hkv);
  const int stage = SH::stage_bytes(cfg->hg);
  int nst = cfg->hg * kRingBytesPerHead / stage;
  nst = nst < 2 ? 2 : nst > kMaxStages ? kMaxStages : nst;
  while (nst > 2 && SH::smem_bytes(cfg->hg, nst, S) > dev.smem_optin) --nst;
  cfg->nst = nst;
  cfg->smem = SH::smem_bytes(cfg->hg, nst, S);
  if (cfg->smem > dev.smem_optin)
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_attention: %zu bytes of shared memory needed",
                    cfg->smem);
  cfg->threads = (cfg->hg + 1 + kMergeWarps) * 32;
  static std::mutex mu;
  static bool attr_set[pa::kMaxDevices] = {};
  struct OccEntry {
    int device, threads;
    size_t smem;
    int occ;
  };
  static OccEntry occ_cache[8];
  static int occ_used = 0, occ_next = 0;
  int occ = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev.device]) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(dev.smem_optin));
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return pa::cuda_fail(e, "cudaFuncSetAttribute");
      attr_set[dev.device] = true;
    }
    for (int i = 0; i < occ_used; ++i) {
      const OccEntry& o = occ_cache[i];
      if (o.device == dev.device && o.threads == cfg->threads && o.smem == cfg->smem) occ = o.occ;
    }
    if (occ == 0) {
      cudaError_t e =
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, cfg->threads, cfg->smem);
      if (e != cudaSuccess) return pa::cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
      occ_cache[occ_next] = OccEntry{dev.device, cfg->threads, cfg->smem, occ};
      occ_next = (occ_next + 1) % 8;
      if (occ_used < 8) ++occ_used;
    }
  }
  if (occ < 1) return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_attention: kernel does not fit an SM");
  long long grid = static_cast<long long>(dev.sm_count) * occ;
  cfg->grid = grid > kMaxGrid ? kMaxGrid : grid;
  return PA_OK;
}

template <int D, int BS, int G, bool KV8, bool PFX = false>
pa_status launch_decode(DecodeParams prm, const pa::DeviceInfo& dev, cudaStream_t stream) {
  using SH = Shape<D, BS, G, KV8>;
  LaunchCfg cfg;
  if (pa_status s = launch_config<D, BS, G, KV8, PFX>(dev, prm.num_seqs, prm.num_kv_heads, &cfg))
    return s;
  prm.hg = cfg.hg;
  prm.nst = cfg.nst;
  CUtensorMap kmap, vmap;
  pa::MapKey kk{dev.device, prm.k_pool, D, BS, prm.num_kv_heads, prm.num_blocks, cfg.hg, SH::TS,
            SH::ESZ, prm.block_stride_bytes};
  pa::MapKey vk{dev.device, prm.v_pool, D, BS, prm.num_kv_heads, prm.num_blocks, cfg.hg, SH::TS,
            SH::ESZ, prm.block_stride_bytes};
  if (pa_status s = pa::pool_tensor_map(kk, &kmap)) return s;
  if (pa_status s = pa::pool_tensor_map(vk, &vmap)) return s;
  // Programmatic dependent launch: the prologue may overlap the tail of the
  // previous kernel on the stream; the kernel waits for it (griddepcontrol)
  // before reading the pool, q or the table.
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(cfg.grid));
  lc.blockDim = dim3(static_cast<unsigned>(cfg.threads));
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&lc, paged_decode_kernel<D, BS, G, KV8, PFX>, prm, kmap, vmap);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return pa::cuda_fail(e, "pa_decode_attention launch");
  pa::count_launch();

  return PA_OK;
}

template <int D, int BS, bool KV8 = false>
pa_status dispatch_g(int G, const DecodeParams& prm, const pa::DeviceInfo& dev, cudaStream_t s) {
  switch (G) {
    case 1: return launch_decode<D, BS, 1, KV8>(prm, dev, s);
    case 2: return launch_decode<D, BS, 2, KV8>(prm, dev, s);
    case 4: return launch_decode<D, BS, 4, KV8>(prm, dev, s);
    case 8: return launch_decode<D, BS, 8, KV8>(prm, dev, s);
  }
  return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_attention: query/KV head ratio %d not in {1,2,4,8}",
                  G);
}

template <int D>
pa_status dispatch_bs(int BS, int G, const DecodeParams& prm, const pa::DeviceInfo& dev,
                      cudaStream_t s) {
  switch (BS) {
    case 8: return dispatch_g<D, 8>(G, prm, dev, s);
    case 16: return dispatch_g<D, 16>(G, prm, dev, s);
    case 32: return dispatch_g<D, 32>(G, prm, dev, s);
  }
  return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_attention: block_size %d not in {8,16,32}", BS);
}

// Launch shape without launching (the allocation-free entry point sizes its
// scratch from the grid).
pa_status launch_config_any(int D, int BS, int G, const pa::DeviceInfo& dev, int S, int Hkv,
                            LaunchCfg* cfg) {
#define PA_CFG_CASE(d, bs, g) \
  if (D == d && BS == bs && G == g) return launch_config<d, bs, g>(dev, S, Hkv, cfg);
#define PA_CFG_G(d, bs) PA_CFG_CASE(d, bs, 1) PA_CFG_CASE(d, bs, 2) PA_CFG_CASE(d, bs, 4) \
  PA_CFG_CASE(d, bs, 8)
  PA_CFG_G(64, 8) PA_CFG_G(64, 16) PA_CFG_G(64, 32)
  PA_CFG_G(128, 8) PA_CFG_G(128, 16) PA_CFG_G(128, 32)
#undef PA_CFG_G
#undef PA_CFG_CASE
  return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_attention: unsupported shape");
}

// Workspace of the shared-prefix call: the regular layout, then one record per
// (sequence, KV head) for segments streamed whole, then the prefix chunks'
// records.
// Regions are counted in whole records from the start of the record area, so
// every record index addresses a record-aligned slot.
struct PfxLayout {
  Layout base;
  long long own_rec = 0, pfx_rec = 0;  // first record of each region
  size_t total = 0;
};
PfxLayout shared_prefix_layout(int S, int Hq, int Hkv, int D, int MB, int P) {
  PfxLayout w;
  w.base = workspace_layout(S, Hq, Hkv, D, MB, 0);
  const int hg = head_group(Hkv);
  const size_t rec = static_cast<size_t>(rec_floats(Hq / Hkv, D)) * 4;
  const long long kmax = pa::max_prefix_chunks();
  const long long cmax = P < kmax ? (P > 0 ? P : 1) : kmax;
  w.own_rec = 2 * max_chunks(S, Hkv / hg, MB, 0) * hg;  // after the chunk records
  w.pfx_rec = w.own_rec + static_cast<long long>(S) * Hkv;
  const long long nrec = w.pfx_rec + cmax * S * Hkv;
  w.total = w.base.records + round256(static_cast<size_t>(nrec) * rec);
  if (w.total < w.base.total) w.total = w.base.total;
  return w;
}

pa_status check_decode_shape(int S, int Hq, int Hkv, int D, int BS, int MB, int part_tokens) {
  if (S < 0 || Hq <= 0 || Hkv <= 0 || MB <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: seqs=%d q_heads=%d kv_heads=%d "
                    "max_blocks=%d", S, Hq, Hkv, MB);
  if (Hq % Hkv) return pa::fail(PA_ERR_INVALID_ARG, "q_heads %d not a multiple of kv_heads %d", Hq, Hkv);
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return pa::fail(PA_ERR_UNSUPPORTED, "query/KV head ratio %d not in {1,2,4,8}", G);
  if (D != 64 && D != 128) return pa::fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64,128}", D);
  if (BS != 8 && BS != 16 && BS != 32)
    return pa::fail(PA_ERR_UNSUPPORTED, "block_size %d not in {8,16,32}", BS);
  if (S > kMaxSeqs) return pa::fail(PA_ERR_UNSUPPORTED, "num_seqs %d > %d", S, kMaxSeqs);
  if (part_tokens < 0 || part_tokens % BS)
    return pa::fail(PA_ERR_INVALID_ARG,
                    "partition_tokens %d must be 0 or a positive multiple of block_size",
                    part_tokens);
  if (static_cast<long long>(MB) * BS > INT32_MAX)
    return pa::fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq * block_size exceeds int32");
  // block-stream positions are 32-bit in the kernel
  if (static_cast<long long>(S) * (Hkv / head_group(Hkv)) * MB >= (1ll << 31))
    return pa::fail(PA_ERR_UNSUPPORTED,
                    "num_seqs x KV head groups x max_blocks_per_seq must stay below 2^31");
  // the chunks one sequence can span must fit the arrival count of a counter word
  const long long cap = part_tokens / BS;
  const long long span = cap > 0 ? (MB + cap - 1) / cap + 1 : kMaxGrid;
  if (span >= (1ll << kArrivalBits))
    return pa::fail(PA_ERR_UNSUPPORTED,
                    "partition_tokens %d splits a sequence of %d blocks into too many chunks",
                    part_tokens, MB);
  return PA_OK;
}


// --- fixed scratch for the entry point that allocates nothing ----------------
// Some callers cannot hand this library a workspace: every byte of device
// memory they own is already given to their KV pool and their own allocator,
// and calling cudaMalloc on the decode path (which also synchronises the
// device) is not an option for them. For those callers the scratch lives in a
// file-scope device array of fixed size instead. Every GPU that loads libpa
// holds these 16 MiB until the process exits.
constexpr size_t kFixedScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_pa_fixed_scratch[kFixedScratchBytes];

// Device address of the fixed scratch on the current device, resolved once
// per device (the host-side symbol is only a stand-in, never a device
// address). Returns nullptr with a recorded message on failure.
unsigned char* fixed_scratch_address(int device) {
  static std::mutex mu;
  static unsigned char* addr[pa::kMaxDevices] = {};
  if (!pa::device_slot_ok(device)) {
    pa::fail(PA_ERR_UNSUPPORTED, "fixed decode scratch: device index %d", device);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_pa_fixed_scratch);
    if (e != cudaSuccess) {
      pa::cuda_fail(e, "cudaGetSymbolAddress(fixed decode scratch)");
      return nullptr;
    }
    addr[device] = static_cast<unsigned char*>(ptr);
  }
  return addr[device];
}

}  // namespace

namespace pa {

// --- TMA descriptors of the pools -------------------------------------------
// A 4-D tensor map over a pool seen as (dim, token, KV head, block) — the
// token stride (Hkv*D*2 bytes) is larger than the head stride (D*2), and the
// block stride is the pool's (a dense block, or two for the one-pool record
// layout whose records hold a block's K and then its V) — with box
// {64, tokens per stage, HG, 1} and the 128-byte swizzle: one copy moves one
// 64-dimension half of HG heads of a block, landing as [head][token][128 B].
// Encoding costs a few microseconds of host time, so the last few maps are
// cached by (device, pointer, shape).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

pa_status pool_tensor_map(const MapKey& key, CUtensorMap* out) {
  static std::mutex mu;
  static EncodeTiledFn encode = nullptr;
  constexpr int kCache = 8;
  static MapKey keys[kCache];
  static CUtensorMap maps[kCache];
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (keys[i] == key) {
      *out = maps[i];
      return PA_OK;
    }
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(key.D), static_cast<cuuint64_t>(key.BS),
                              static_cast<cuuint64_t>(key.Hkv), static_cast<cuuint64_t>(key.NB)};
  const cuuint64_t e = static_cast<cuuint64_t>(key.esz);
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(key.Hkv) * key.D * e,   // token
                                 static_cast<cuuint64_t>(key.D) * e,             // KV head
                                 static_cast<cuuint64_t>(key.stride)};                  // block
  // the box's inner extent is one 128-byte line: 64 fp16 or 128 E4M3 values
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / key.esz),
                             static_cast<cuuint32_t>(key.ts), static_cast<cuuint32_t>(key.hg), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMap m;
  CUresult r = encode(&m, key.esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      4, const_cast<void*>(key.ptr), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a pool of %d blocks",
                    static_cast<int>(r), key.NB);
  keys[next] = key;
  maps[next] = m;
  next = (next + 1) % kCache;
  if (used < kCache) ++used;
  *out = m;
  return PA_OK;
}

}  // namespace pa

extern "C" {

size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_blocks_per_seq, int partition_tokens) {
  if (check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq, partition_tokens) != PA_OK)
    return 0;
  return workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                          partition_tokens / block_size)
      .total;
}

pa_status pa_decode_workspace_init(void* workspace, size_t workspace_bytes, int num_seqs,
                                   int num_kv_heads, pa_stream_t stream) {
  if (num_seqs < 0 || num_kv_heads <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "workspace_init: seqs=%d kv_heads=%d", num_seqs,
                    num_kv_heads);
  const size_t need = static_cast<size_t>(num_seqs) * num_kv_heads * 8;
  if (need == 0) return pa::ok();
  if (!workspace || workspace_bytes < need)
    return pa::fail(PA_ERR_INVALID_ARG, "workspace_init: %zu bytes < %zu", workspace_bytes, need);
  cudaError_t e = cudaMemsetAsync(workspace, 0, need, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return pa::cuda_fail(e, "workspace_init");
  return pa::ok();
}

// Host checks shared by both decode entry points.
static pa_status check_decode_call(const char* fn, const pa_half* q, const pa_half* k_pool,
                                   const pa_half* v_pool, const int32_t* block_table,
                                   const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int max_blocks_per_seq, int num_blocks,
                                   int64_t pool_block_stride, int esz, float scale,
                                   const pa_half* out, int partition_tokens,
                                   long long* stride_bytes) {
  if (pa_status s = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                       max_blocks_per_seq, partition_tokens))
    return s;
  if (num_blocks <= 0 || static_cast<long long>(num_blocks) * block_size > INT32_MAX)
    return pa::fail(PA_ERR_INVALID_ARG, "%s: num_blocks %d", fn, num_blocks);
  int64_t stride = 0;
  if (pa_status s = pa::resolve_block_stride(
          fn, pool_block_stride, static_cast<int64_t>(block_size) * num_kv_heads * head_dim, esz,
          &stride))
    return s;
  *stride_bytes = stride * esz;
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return pa::fail(PA_ERR_INVALID_ARG, "%s: scale is not finite", fn);
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out)
    return pa::fail(PA_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (!pa::aligned16(q) || !pa::aligned16(k_pool) || !pa::aligned16(v_pool) ||
      !pa::aligned16(out) || (reinterpret_cast<uintptr_t>(block_table) & 3) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  return PA_OK;
}

// q, the table, the lengths and the output may be device memory or pinned
// host memory, which the kernels then read and write through its device
// mapping (zero-copy over the CPU-GPU link); the pools must be device memory
// (the kernels reach them through TMA).
static pa_status resolve_io(const char* fn, const pa_half*& q, const void* k_pool,
                            const void* v_pool, const int32_t*& block_table,
                            const int32_t*& seq_lens, pa_half*& out) {
  if (pa_status s = pa::device_only(fn, k_pool)) return s;
  if (pa_status s = pa::device_only(fn, v_pool)) return s;
  if (pa_status s = pa::device_in(fn, q)) return s;
  if (pa_status s = pa::device_in(fn, block_table)) return s;
  if (pa_status s = pa::device_in(fn, seq_lens)) return s;
  return pa::device_in(fn, out);
}

static DecodeParams make_params(const pa_half* q, const pa_half* k_pool, const pa_half* v_pool,
                                const int32_t* block_table, const int32_t* seq_lens,
                                int num_seqs, int num_q_heads, int num_kv_heads,
                                int max_blocks_per_seq, int num_blocks, long long stride_bytes,
                                float scale, pa_half* out, unsigned char* ws, const Layout& lay,
                                int cap_blocks) {
  DecodeParams prm;
  prm.q = reinterpret_cast<const __half*>(q);
  prm.k_pool = reinterpret_cast<const __half*>(k_pool);
  prm.v_pool = reinterpret_cast<const __half*>(v_pool);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.k_scale = nullptr;
  prm.v_scale = nullptr;
  prm.pfx_blocks = 0;
  prm.pfx_chunks = 0;
  prm.pfx_rec_base = 0;
  prm.pfx_own_base = 0;
  prm.out = reinterpret_cast<__half*>(out);
  prm.records = reinterpret_cast<float*>(ws + lay.records);
  prm.counters = reinterpret_cast<unsigned long long*>(ws + lay.counters);
  prm.tag = next_call_tag();
  prm.err = nullptr;
  prm.num_seqs = num_seqs;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_blocks = num_blocks;
  prm.cap_blocks = cap_blocks;
  prm.hg = 0;   // set by the launch
  prm.nst = 0;  // set by the launch
  prm.qscale = scale * kLog2e;
  prm.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  prm.block_stride_bytes = stride_bytes;
  prm.k_new = nullptr;
  prm.v_new = nullptr;
  prm.slot_mapping = nullptr;
  prm.block_stride = stride_bytes / 2;
  return prm;
}

pa_status pa_decode_attention(const pa_half* q, const pa_half* k_pool, const pa_half* v_pool,
                              const int32_t* block_table, const int32_t* seq_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks_per_seq, int num_blocks, int64_t pool_block_stride,
                              float scale, pa_half* out, void* workspace, size_t workspace_bytes,
                              int partition_tokens, pa_stream_t stream) {
  long long stride_bytes = 0;
  if (pa_status s = check_decode_call("pa_decode_attention", q, k_pool, v_pool, block_table,
                                      seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      block_size, max_blocks_per_seq, num_blocks,
                                      pool_block_stride, 2, scale, out, partition_tokens,
                                      &stride_bytes))
    return s;
  if (num_seqs == 0) return pa::ok();
  if (pa_status s = resolve_io("pa_decode_attention", q, k_pool, v_pool, block_table, seq_lens,
                               out))
    return s;
  if (workspace) {
    if (pa_status s = pa::device_only("pa_decode_attention(workspace)", workspace)) return s;
  }
  if (!workspace) return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: NULL workspace");
  if (!pa::aligned16(workspace))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: misaligned workspace");
  const int cap_blocks = partition_tokens / block_size;
  const Layout lay = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq, cap_blocks);
  if (workspace_bytes < lay.total)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: workspace %zu < %zu bytes",
                    workspace_bytes, lay.total);
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  DecodeParams prm = make_params(q, k_pool, v_pool, block_table, seq_lens, num_seqs, num_q_heads,
                                 num_kv_heads, max_blocks_per_seq, num_blocks, stride_bytes,
                                 scale, out, static_cast<unsigned char*>(workspace), lay,
                                 cap_blocks);
  prm.err = pa::device_error_word();
  if (!prm.err) return PA_ERR_CUDA;
  const int G = num_q_heads / num_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  pa_status st = head_dim == 64 ? dispatch_bs<64>(block_size, G, prm, dev, s)
                                : dispatch_bs<128>(block_size, G, prm, dev, s);
  return st == PA_OK ? pa::ok() : st;
}

pa_status pa_decode_append_attention(const pa_half* q, const pa_half* k_new,
                                     const pa_half* v_new, const int32_t* slot_mapping,
                                     pa_half* k_pool, pa_half* v_pool,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int max_blocks_per_seq,
                                     int num_blocks, int64_t pool_block_stride, float scale,
                                     pa_half* out, void* workspace, size_t workspace_bytes,
                                     int partition_tokens, pa_stream_t stream) {
  const char* fn = "pa_decode_append_attention";
  long long stride_bytes = 0;
  if (pa_status s = check_decode_call(fn, q, k_pool, v_pool, block_table, seq_lens, num_seqs,
                                      num_q_heads, num_kv_heads, head_dim, block_size,
                                      max_blocks_per_seq, num_blocks, pool_block_stride, 2, scale,
                                      out, partition_tokens, &stride_bytes))
    return s;
  if (num_seqs == 0) return pa::ok();
  if (!k_new || !v_new || !slot_mapping)
    return pa::fail(PA_ERR_INVALID_ARG, "%s: NULL k_new, v_new or slot_mapping", fn);
  if (!pa::aligned16(k_new) || !pa::aligned16(v_new) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "%s: misaligned k_new, v_new or slot_mapping", fn);
  if (pa_status s = pa::check_pools_disjoint(
          fn, k_pool, v_pool, num_blocks, stride_bytes,
          static_cast<int64_t>(block_size) * num_kv_heads * head_dim * 2))
    return s;
  const pa_half* qd = q;
  const int32_t* table = block_table;
  const int32_t* lens = seq_lens;
  pa_half* outd = out;
  if (pa_status s = resolve_io(fn, qd, k_pool, v_pool, table, lens, outd)) return s;
  if (pa_status s = pa::device_in("pa_decode_append_attention(k_new)", k_new)) return s;
  if (pa_status s = pa::device_in("pa_decode_append_attention(v_new)", v_new)) return s;
  if (pa_status s = pa::device_in("pa_decode_append_attention(slot_mapping)", slot_mapping))
    return s;
  if (!workspace) return pa::fail(PA_ERR_INVALID_ARG, "%s: NULL workspace", fn);
  if (pa_status s = pa::device_only("pa_decode_append_attention(workspace)", workspace)) return s;
  if (!pa::aligned16(workspace)) return pa::fail(PA_ERR_INVALID_ARG, "%s: misaligned workspace", fn);
  const int cap_blocks = partition_tokens / block_size;
  const Layout lay = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq, cap_blocks);
  if (workspace_bytes < lay.total)
    return pa::fail(PA_ERR_INVALID_ARG, "%s: workspace %zu < %zu bytes", fn, workspace_bytes,
                    lay.total);
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  DecodeParams prm = make_params(qd, k_pool, v_pool, table, lens, num_seqs, num_q_heads,
                                 num_kv_heads, max_blocks_per_seq, num_blocks, stride_bytes,
                                 scale, outd, static_cast<unsigned char*>(workspace), lay,
                                 cap_blocks);
  prm.err = pa::device_error_word();
  if (!prm.err) return PA_ERR_CUDA;
  prm.k_new = reinterpret_cast<const __half*>(k_new);
  prm.v_new = reinterpret_cast<const __half*>(v_new);
  prm.slot_mapping = slot_mapping;
  const int G = num_q_heads / num_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  pa_status st = head_dim == 64 ? dispatch_bs<64>(block_size, G, prm, dev, s)
                                : dispatch_bs<128>(block_size, G, prm, dev, s);
  return st == PA_OK ? pa::ok() : st;
}

pa_status pa_decode_attention_fp8(const pa_half* q, const uint8_t* k_pool, const uint8_t* v_pool,
                                  const float* k_scale, const float* v_scale,
                                  const int32_t* block_table, const int32_t* seq_lens,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_blocks_per_seq, int num_blocks,
                                  int64_t pool_block_stride, float scale, pa_half* out,
                                  void* workspace, size_t workspace_bytes, int partition_tokens,
                                  pa_stream_t stream) {
  const pa_half* kp = reinterpret_cast<const pa_half*>(k_pool);
  const pa_half* vp = reinterpret_cast<const pa_half*>(v_pool);
  long long stride_bytes = 0;
  if (pa_status s = check_decode_call("pa_decode_attention_fp8", q, kp, vp, block_table, seq_lens,
                                      num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                      max_blocks_per_seq, num_blocks, pool_block_stride, 1, scale,
                                      out, partition_tokens, &stride_bytes))
    return s;
  if (head_dim != 128 || (block_size != 16 && block_size != 32))
    return pa::fail(PA_ERR_UNSUPPORTED,
                    "pa_decode_attention_fp8: head_dim %d / block_size %d (fp8 pools support "
                    "head_dim 128 and block_size 16 or 32)", head_dim, block_size);
  if (num_seqs == 0) return pa::ok();
  if (pa_status s = resolve_io("pa_decode_attention_fp8", q, k_pool, v_pool, block_table,
                               seq_lens, out))
    return s;
  if (pa_status s = pa::device_in("pa_decode_attention_fp8(k_scale)", k_scale)) return s;
  if (workspace) {
    if (pa_status s = pa::device_only("pa_decode_attention_fp8(workspace)", workspace)) return s;
  }
  if (pa_status s = pa::device_in("pa_decode_attention_fp8(v_scale)", v_scale)) return s;
  if (!k_scale || !v_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3) ||
      (reinterpret_cast<uintptr_t>(v_scale) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention_fp8: NULL or misaligned scales");
  if (!workspace) return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention_fp8: NULL workspace");
  if (!pa::aligned16(workspace))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention_fp8: misaligned workspace");
  const int cap_blocks = partition_tokens / block_size;
  const Layout lay = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq, cap_blocks);
  if (workspace_bytes < lay.total)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention_fp8: workspace %zu < %zu bytes",
                    workspace_bytes, lay.total);
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  DecodeParams prm = make_params(q, kp, vp, block_table, seq_lens, num_seqs, num_q_heads,
                                 num_kv_heads, max_blocks_per_seq, num_blocks, stride_bytes,
                                 scale, out, static_cast<unsigned char*>(workspace), lay,
                                 cap_blocks);
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.err = pa::device_error_word();
  if (!prm.err) return PA_ERR_CUDA;
  const int G = num_q_heads / num_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  pa_status st = block_size == 16 ? dispatch_g<128, 16, true>(G, prm, dev, s)
                                  : dispatch_g<128, 32, true>(G, prm, dev, s);
  return st == PA_OK ? pa::ok() : st;
}

size_t pa_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                                int head_dim, int block_size,
                                                int max_blocks_per_seq, int num_prefix_blocks) {
  if (check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq, 0) != PA_OK)
    return 0;
  if (num_prefix_blocks < 0 || num_prefix_blocks > max_blocks_per_seq) return 0;
  return shared_prefix_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                              num_prefix_blocks)
      .total;
}

pa_status pa_decode_attention_shared_prefix(
    const pa_half* q, const pa_half* k_pool, const pa_half* v_pool, const int32_t* prefix_blocks,
    int num_prefix_blocks, const int32_t* block_table, const int32_t* seq_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
    int num_blocks, int64_t pool_block_stride, float scale, pa_half* out, void* workspace,
    size_t workspace_bytes, pa_stream_t stream) {
  long long stride_bytes = 0;
  if (pa_status s = check_decode_call("pa_decode_attention_shared_prefix", q, k_pool, v_pool,
                                      block_table, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                                      head_dim, block_size, max_blocks_per_seq, num_blocks,
                                      pool_block_stride, 2, scale, out, 0, &stride_bytes))
    return s;
  if (head_dim != 128 || (block_size != 16 && block_size != 32))
    return pa::fail(PA_ERR_UNSUPPORTED,
                    "pa_decode_attention_shared_prefix: head_dim %d / block_size %d (supported: "
                    "head_dim 128, block_size 16 or 32)", head_dim, block_size);
  if (num_prefix_blocks < 0 || num_prefix_blocks > max_blocks_per_seq)
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention_shared_prefix: num_prefix_blocks %d not in [0, %d]",
                    num_prefix_blocks, max_blocks_per_seq);
  if (num_seqs == 0) return pa::ok();
  if (pa_status s = resolve_io("pa_decode_attention_shared_prefix", q, k_pool, v_pool,
                               block_table, seq_lens, out))
    return s;
  if (pa_status s = pa::device_in("pa_decode_attention_shared_prefix(prefix_blocks)",
                                  prefix_blocks))
    return s;
  if (workspace) {
    if (pa_status s = pa::device_only("pa_decode_attention_shared_prefix(workspace)", workspace))
      return s;
  }
  if (num_prefix_blocks > 0 &&
      (!prefix_blocks || (reinterpret_cast<uintptr_t>(prefix_blocks) & 3)))
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention_shared_prefix: NULL or misaligned prefix_blocks");
  if (!workspace || !pa::aligned16(workspace))
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention_shared_prefix: NULL or misaligned workspace");
  const PfxLayout lay = shared_prefix_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, num_prefix_blocks);
  if (workspace_bytes < lay.total)
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention_shared_prefix: workspace %zu < %zu bytes",
                    workspace_bytes, lay.total);
  if (num_prefix_blocks == 0)
    return pa_decode_attention(q, k_pool, v_pool, block_table, seq_lens, num_seqs, num_q_heads,
                               num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                               num_blocks, pool_block_stride, scale, out, workspace,
                               workspace_bytes, 0, stream);
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  const int G = num_q_heads / num_kv_heads;
  const int P = num_prefix_blocks;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const size_t rec_bytes = static_cast<size_t>(rec_floats(G, head_dim)) * 4;
  // the suffix pass: the table past the prefix's columns, lengths past its tokens
  DecodeParams prm = make_params(q, k_pool, v_pool, block_table + P, seq_lens, num_seqs,
                                 num_q_heads, num_kv_heads, max_blocks_per_seq, num_blocks,
                                 stride_bytes, scale, out, ws, lay.base, 0);
  prm.err = pa::device_error_word();
  if (!prm.err) return PA_ERR_CUDA;
  prm.pfx_blocks = P;
  prm.pfx_own_base = lay.own_rec;
  prm.pfx_rec_base = lay.pfx_rec;
  pa::SharedPrefixCall call;
  call.q = q;
  call.prefix_blocks = prefix_blocks;
  call.records = reinterpret_cast<float*>(ws + lay.base.records + lay.pfx_rec * rec_bytes);
  call.err = prm.err;
  call.num_seqs = num_seqs;
  call.num_q_heads = num_q_heads;
  call.num_kv_heads = num_kv_heads;
  call.head_dim = head_dim;
  call.block_size = block_size;
  call.max_blocks = max_blocks_per_seq;
  call.num_blocks = num_blocks;
  call.prefix_blocks_n = P;
  call.qscale = scale * kLog2e;
  call.block_table = prm.block_table - P;  // the whole table (prm's starts past the prefix)
  call.seq_lens = prm.seq_lens;
  call.k_pool = k_pool;
  call.v_pool = v_pool;
  call.block_stride_bytes = stride_bytes;
  call.out = prm.out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool suffix_pass = false;
  int chunks = 0;
  pa_status st = pa::launch_shared_prefix(call, dev, s, &suffix_pass, &chunks);
  if (st == PA_OK && suffix_pass) {
    // the rest of each sequence, folding the prefix chunks' records
    prm.pfx_chunks = chunks;
#define PA_PFX_CASE(bs, g) \
    if (block_size == bs && G == g) st = launch_decode<128, bs, g, false, true>(prm, dev, s); else
    PA_PFX_CASE(16, 1) PA_PFX_CASE(16, 2) PA_PFX_CASE(16, 4) PA_PFX_CASE(16, 8)
    PA_PFX_CASE(32, 1) PA_PFX_CASE(32, 2) PA_PFX_CASE(32, 4) PA_PFX_CASE(32, 8)
    st = pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_attention_shared_prefix: unsupported shape");
#undef PA_PFX_CASE
  }
  return st == PA_OK ? pa::ok() : st;
}

pa_status pa_decode_attention_fixed_scratch(const pa_half* q, const pa_half* k_pool,
                                            const pa_half* v_pool, const int32_t* block_table,
                                            const int32_t* seq_lens, int num_seqs,
                                            int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, int max_blocks_per_seq,
                                            int num_blocks, int64_t pool_block_stride,
                                            float scale, pa_half* out, int partition_tokens,
                                            pa_stream_t stream) {
  long long stride_bytes = 0;
  if (pa_status s = check_decode_call("pa_decode_attention_fixed_scratch", q, k_pool, v_pool,
                                      block_table, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                                      head_dim, block_size, max_blocks_per_seq, num_blocks,
                                      pool_block_stride, 2, scale, out, partition_tokens,
                                      &stride_bytes))
    return s;
  if (num_seqs == 0) return pa::ok();
  if (pa_status s = resolve_io("pa_decode_attention_fixed_scratch", q, k_pool, v_pool,
                               block_table, seq_lens, out))
    return s;
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  const int G = num_q_heads / num_kv_heads;
  LaunchCfg cfg;
  if (pa_status s = launch_config_any(head_dim, block_size, G, dev, num_seqs, num_kv_heads, &cfg))
    return s;
  // scratch this call needs: arrival counters, then two partial records per
  // chunk (one per CTA of this grid, or more with a partition cap) and KV
  // head of the group
  const int cap_blocks = partition_tokens / block_size;
  long long chunks = cfg.grid;
  if (cap_blocks > 0) {
    const long long blocks =
        static_cast<long long>(num_seqs) * (num_kv_heads / cfg.hg) * max_blocks_per_seq;
    const long long capped = (blocks + cap_blocks - 1) / cap_blocks;
    if (capped > chunks) chunks = capped;
  }
  Layout lay;
  lay.counters = 0;
  lay.records = round256(static_cast<size_t>(num_seqs) * num_kv_heads * 8);
  lay.total = lay.records + static_cast<size_t>(2 * chunks) * cfg.hg *
                                rec_floats(G, head_dim) * sizeof(float);
  const size_t need = lay.total;
  if (need > kFixedScratchBytes)
    return pa::fail(PA_ERR_UNSUPPORTED,
                    "pa_decode_attention_fixed_scratch: this shape needs %zu bytes of scratch; "
                    "the fixed scratch holds %zu (use pa_decode_attention with a workspace)",
                    need, kFixedScratchBytes);
  unsigned char* ws = fixed_scratch_address(dev.device);
  if (!ws) return pa::device_slot_ok(dev.device) ? PA_ERR_CUDA : PA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the last call left. A call cut short by a
  // timeout leaves arrival counts under its tag, and a replayed graph reuses
  // its tag, so the counters are cleared here on every call (no caller can
  // clear this array).
  if (cudaError_t e = cudaMemsetAsync(ws + lay.counters, 0,
                                      static_cast<size_t>(num_seqs) * num_kv_heads * 8, s))
    return pa::cuda_fail(e, "pa_decode_attention_fixed_scratch: clearing the counters");
  DecodeParams prm = make_params(q, k_pool, v_pool, block_table, seq_lens, num_seqs, num_q_heads,
                                 num_kv_heads, max_blocks_per_seq, num_blocks, stride_bytes,
                                 scale, out, ws, lay, cap_blocks);
  prm.err = pa::device_error_word();
  if (!prm.err) return PA_ERR_CUDA;
  pa_status st = head_dim == 64 ? dispatch_bs<64>(block_size, G, prm, dev, s)
                                : dispatch_bs<128>(block_size, G, prm, dev, s);
  return st == PA_OK ? pa::ok() : st;
}

pa_status pa_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns == 0 ? kWaitLimitNs : limit_ns, std::memory_order_relaxed);
  return pa::ok();
}

}  // extern "C"
