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
//   * Work item = (sequence, KV head, partition of `partition_tokens` tokens).
//     All G query heads of a KV head are served by one item, so every K/V byte
//     is read from HBM once per step (GQA head-group reuse).
//   * Persistent grid (SMs x resident CTAs). Items are numbered KV-head-fastest
//     so CTAs running side by side stream neighbouring rows of the same blocks.
//     Each CTA derives the item list from a prefix sum of per-sequence
//     partition counts held in shared memory (no host-side plan, no extra
//     launch).
//   * Warp specialisation: one producer warp walks the CTA's items, reads the
//     block-table entries of an item with one coalesced load, and issues one
//     bulk async copy (cp.async.bulk, completion counted on an mbarrier) per K
//     row and per V row of each block into a ring of shared-memory stages.
//     Four consumer warps take the stages round-robin.
//   * Consumer math: a row of head_dim fp16 values is split over 8 or 16 lanes
//     (16-byte vector reads from shared memory, conflict-free); each lane
//     keeps q (pre-scaled by scale*log2 e) and its slice of the fp32
//     accumulators in registers and uses the packed fp32 FMA (fma.rn.f32x2).
//     Dot products are finished with xor-shuffles inside the lane group, and
//     the softmax is the online (running max / running sum) form in base 2.
//   * End of an item: warp partial states are merged with shuffles, then
//     across warps through shared memory. An unsplit sequence writes fp16
//     output directly. A split sequence writes its (max, sum, acc) partial to
//     the workspace; the last CTA to finish a (sequence, KV head) — found with
//     an atomic arrival counter, never a spin — merges all partials with the
//     log-sum-exp rule and writes the output, then resets the counter.
//   * Every wait is bounded (about one second of %globaltimer); on expiry the
//     kernel records PA_DEVERR_TIMEOUT, stops issuing copies, drains the copies
//     already in flight (again bounded) and finishes without faulting.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kDefaultPartitionTokens = 256;
constexpr int kMaxSeqs = 16384;
constexpr int kRingBytes = 64 * 1024;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ PTX ---
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bulk async copy global -> this CTA's shared memory, completion on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// d = a * b + c on both halves (packed fp32 FMA, sm_100+).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Warp-collective bounded wait on an mbarrier phase. Every lane polls (so
// each lane itself observes the phase completion); the give-up decision is
// taken by lane 0 and broadcast, so the result is warp-uniform. Returns false
// if the phase does not complete within the time limit (the CTA is then
// flagged as aborted and PA_DEVERR_TIMEOUT recorded once) or if the CTA was
// already aborted.
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, int32_t* err) {
  const int lane = threadIdx.x & 31;
  unsigned long long t0 = 0;
  for (int iter = 0;; ++iter) {
    const bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    int give_up = 0;
    if (lane == 0) {
      if (iter == 0) {
        t0 = global_ns();
      } else if (*abort_flag) {
        give_up = 1;
      } else if (global_ns() - t0 > kWaitLimitNs) {
        if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) atomicOr(err, PA_DEVERR_TIMEOUT);
        give_up = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}

// ------------------------------------------------------------- shapes ---
template <int D, int BS, int G>
struct Shape {
  // lanes sharing one K/V row: keep G * (D / LPR) accumulators <= 64 floats
  static constexpr int LPR = (G * (D / 8) <= 64) ? 8 : 16;
  static constexpr int SG = 32 / LPR;      // row groups per warp
  static constexpr int DPL = D / LPR;      // dims per lane
  static constexpr int NCH = DPL / 8;      // 16-byte chunks per lane per row
  static constexpr int H2 = DPL / 2;       // float2 per lane per head
  static constexpr int TPS = BS / SG;      // rows per group per block
  static constexpr int TB0 = (16 / G) > 0 ? (16 / G) : 1;
  static constexpr int TB = TPS < TB0 ? TPS : TB0;  // rows per softmax update
  static constexpr int NBATCH = TPS / TB;
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int TILE_BYTES = BS * ROW_BYTES;  // K (or V) rows of one block, one head
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int NST = (kRingBytes / STAGE_BYTES) > 4 ? (kRingBytes / STAGE_BYTES) : 4;
  static_assert(D % (LPR * 8) == 0, "head_dim must split into 16-byte chunks per lane");
  static_assert(BS % SG == 0 && TPS % TB == 0, "block size must split over row groups");
  // shared-memory layout (bytes)
  static constexpr int OFF_FULL = 0;
  static constexpr int OFF_EMPTY = OFF_FULL + NST * 8;
  static constexpr int OFF_FLAGS = OFF_EMPTY + NST * 8;           // abort, is_last, wsum[8]
  static constexpr int OFF_RING = ((OFF_FLAGS + 64) + 127) / 128 * 128;
  static constexpr int OFF_MACC = OFF_RING + NST * STAGE_BYTES;  // float [NC][G][D]
  static constexpr int OFF_MML = OFF_MACC + kConsumerWarps * G * D * 4;  // float [NC][G][2]
  static constexpr int OFF_PREFIX = OFF_MML + kConsumerWarps * G * 2 * 4;
  static size_t smem_bytes(int num_seqs) {
    return static_cast<size_t>(OFF_PREFIX) + static_cast<size_t>(num_seqs + 1) * 4;
  }
};

struct DecodeParams {
  const __half* q;
  const __half* k_pool;
  const __half* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  __half* out;
  int32_t* counters;  // [S][Hkv]
  float* part_ml;     // [S][Hkv][max_splits][G][2]
  float* part_acc;    // [S][Hkv][max_splits][G][D]
  int32_t* err;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int max_blocks;
  int num_blocks;
  int part_blocks;  // blocks per partition (<= 32)
  int max_splits;
  float qscale;  // scale * log2(e)
};

__device__ __forceinline__ int clamp_len(int L, int cap, int32_t* err) {
  if (L < 0 || L > cap) {
    atomicOr(err, PA_DEVERR_BAD_LEN);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

struct Item {
  int seq, split, kvh;
};

// Item w -> (sequence, partition, KV head), KV head fastest.
__device__ __forceinline__ Item decode_item(long long w, int hkv, const int* prefix, int S) {
  Item it;
  it.kvh = static_cast<int>(w % hkv);
  const int u = static_cast<int>(w / hkv);
  int lo = 0, hi = S;  // largest i with prefix[i] <= u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= u) lo = mid;
    else hi = mid;
  }
  it.seq = lo;
  it.split = u - prefix[lo];
  return it;
}

template <int D, int BS, int G>
__global__ void __launch_bounds__(kThreads, 2) paged_decode_kernel(const DecodeParams p) {
  using SH = Shape<D, BS, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + SH::OFF_FULL);
  uint64_t* empty_bar = reinterpret_cast<uint64_t*>(smem + SH::OFF_EMPTY);
  int* flags = reinterpret_cast<int*>(smem + SH::OFF_FLAGS);
  volatile int* abort_flag = flags;
  unsigned char* ring = smem + SH::OFF_RING;
  float* m_acc = reinterpret_cast<float*>(smem + SH::OFF_MACC);
  float* m_ml = reinterpret_cast<float*>(smem + SH::OFF_MML);
  int* prefix = reinterpret_cast<int*>(smem + SH::OFF_PREFIX);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.num_seqs;
  const int Hkv = p.num_kv_heads;
  const int cap = p.max_blocks * BS;

  if (tid == 0) {
    for (int s = 0; s < SH::NST; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    flags[0] = 0;
    flags[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- partitions per sequence, exclusive prefix sum in shared memory ----
  for (int i = tid; i < S; i += kThreads) {
    const int L = clamp_len(__ldg(p.seq_lens + i), cap, p.err);
    const int nblk = (L + BS - 1) / BS;
    const int ns = (nblk + p.part_blocks - 1) / p.part_blocks;
    prefix[i + 1] = ns > 0 ? ns : 1;
  }
  if (tid == 0) prefix[0] = 0;
  __syncthreads();
  {
    const int per = (S + kThreads - 1) / kThreads;
    const int lo = min(S, tid * per), hi = min(S, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += prefix[i + 1];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int* wsum = flags + 2;
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int i = lo; i < hi; ++i) {
      run += prefix[i + 1];
      prefix[i + 1] = run;
    }
  }
  __syncthreads();
  const long long total_items = static_cast<long long>(prefix[S]) * Hkv;

  if (warp == kConsumerWarps) {
    // =========================== producer warp ===========================
    uint32_t g = 0;  // ring sequence number
    for (long long w = blockIdx.x; w < total_items; w += gridDim.x) {
      const Item it = decode_item(w, Hkv, prefix, S);
      const int L = min(max(__ldg(p.seq_lens + it.seq), 0), cap);
      const int nblk = (L + BS - 1) / BS;
      const int b0 = it.split * p.part_blocks;
      const int nb = max(0, min(nblk, b0 + p.part_blocks) - b0);
      const int phys_lane =
          lane < nb ? __ldg(p.block_table + static_cast<long long>(it.seq) * p.max_blocks + b0 + lane)
                    : 0;
      for (int j = 0; j < nb; ++j, ++g) {
        const int stage = g % SH::NST;
        const uint32_t use = g / SH::NST;
        const int phys = __shfl_sync(0xffffffffu, phys_lane, j);
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) continue;
        if (use > 0 &&
            !warp_wait_phase(smem_addr(&empty_bar[stage]), (use - 1) & 1, abort_flag, p.err))
          continue;
        const bool bad = phys < 0 || phys >= p.num_blocks;
        const int rows = min(BS, L - (b0 + j) * BS);
        const uint32_t fb = smem_addr(&full_bar[stage]);
        if (lane == 0) {
          if (bad) atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
          mbar_arrive_expect_tx(fb, bad ? 0u : 2u * rows * SH::ROW_BYTES);
        }
        __syncwarp();
        if (!bad) {
          const uint32_t kdst = smem_addr(ring + stage * SH::STAGE_BYTES);
          const long long row0 = static_cast<long long>(phys) * BS;
          for (int c = lane; c < 2 * rows; c += 32) {
            const bool is_v = c >= rows;
            const int r = is_v ? c - rows : c;
            const __half* src =
                (is_v ? p.v_pool : p.k_pool) + ((row0 + r) * Hkv + it.kvh) * static_cast<long long>(D);
            bulk_copy_g2s(kdst + (is_v ? SH::TILE_BYTES : 0) + r * SH::ROW_BYTES, src,
                          SH::ROW_BYTES, fb);
          }
        }
      }
    }
    // After an abort, wait (bounded) for copies still landing in the ring.
    if (*abort_flag) {
      const uint32_t first = g > static_cast<uint32_t>(SH::NST) ? g - SH::NST : 0;
      for (uint32_t gi = first; gi < g; ++gi) {
        const uint32_t bar = smem_addr(&full_bar[gi % SH::NST]);
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(bar, (gi / SH::NST) & 1) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    return;
  }

  // ============================ consumer warps ============================
  const int cw = warp;
  const int grp = lane / SH::LPR;  // row group within the warp
  const int gl = lane % SH::LPR;   // lane within the row group
  const int ct = tid;              // consumer thread index 0..127
  uint32_t g = 0;

  for (long long w = blockIdx.x; w < total_items; w += gridDim.x) {
    const Item it = decode_item(w, Hkv, prefix, S);
    const int L = min(max(__ldg(p.seq_lens + it.seq), 0), cap);
    const int nblk = (L + BS - 1) / BS;
    const int b0 = it.split * p.part_blocks;
    const int nb = max(0, min(nblk, b0 + p.part_blocks) - b0);
    const int nsplit = prefix[it.seq + 1] - prefix[it.seq];
    const int head0 = it.kvh * G;

    // q of the G heads, this lane's dims, pre-scaled into the base-2 domain
    float2 q2[G][SH::H2];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const __half* qrow =
          p.q + (static_cast<long long>(it.seq) * p.num_q_heads + head0 + gg) * static_cast<long long>(D);
#pragma unroll
      for (int c = 0; c < SH::NCH; ++c) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow) + c * SH::LPR + gl);
        const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h[e]);
          q2[gg][c * 4 + e] = make_float2(f.x * p.qscale, f.y * p.qscale);
        }
      }
    }
    float m[G], l[G];
    float2 acc[G][SH::H2];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      m[gg] = -INFINITY;
      l[gg] = 0.f;
#pragma unroll
      for (int e = 0; e < SH::H2; ++e) acc[gg][e] = make_float2(0.f, 0.f);
    }

    for (int j = cw; j < nb; j += kConsumerWarps) {
      const uint32_t gj = g + j;
      const int stage = gj % SH::NST;
      if (!warp_wait_phase(smem_addr(&full_bar[stage]), (gj / SH::NST) & 1, abort_flag, p.err))
        continue;
      const int rows = min(BS, L - (b0 + j) * BS);
      const bool full = rows == BS;
      const unsigned char* kt = ring + stage * SH::STAGE_BYTES;
      const unsigned char* vt = kt + SH::TILE_BYTES;
#pragma unroll
      for (int bt = 0; bt < SH::NBATCH; ++bt) {
        float s[SH::TB][G];
#pragma unroll
        for (int k = 0; k < SH::TB; ++k) {
          const int row = (bt * SH::TB + k) * SH::SG + grp;
          float2 a[G];
#pragma unroll
          for (int gg = 0; gg < G; ++gg) a[gg] = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < SH::NCH; ++c) {
            const uint4 raw =
                *reinterpret_cast<const uint4*>(kt + row * SH::ROW_BYTES + (c * SH::LPR + gl) * 16);
            const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 kf = __half22float2(h[e]);
#pragma unroll
              for (int gg = 0; gg < G; ++gg) a[gg] = ffma2(q2[gg][c * 4 + e], kf, a[gg]);
            }
          }
#pragma unroll
          for (int gg = 0; gg < G; ++gg) s[k][gg] = a[gg].x + a[gg].y;
        }
#pragma unroll
        for (int off = 1; off < SH::LPR; off <<= 1) {
#pragma unroll
          for (int k = 0; k < SH::TB; ++k)
#pragma unroll
            for (int gg = 0; gg < G; ++gg) s[k][gg] += __shfl_xor_sync(0xffffffffu, s[k][gg], off);
        }
        // online softmax update (base 2)
        float pr[SH::TB][G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < SH::TB; ++k) {
            const bool valid = full || ((bt * SH::TB + k) * SH::SG + grp) < rows;
            if (valid) mx = fmaxf(mx, s[k][gg]);
          }
          const float mn = fmaxf(m[gg], mx);
          const float mu = mn == -INFINITY ? 0.f : mn;
          const float alpha = fast_exp2(m[gg] - mu);
          float ps = 0.f;
#pragma unroll
          for (int k = 0; k < SH::TB; ++k) {
            const bool valid = full || ((bt * SH::TB + k) * SH::SG + grp) < rows;
            pr[k][gg] = valid ? fast_exp2(s[k][gg] - mu) : 0.f;
            ps += pr[k][gg];
          }
          l[gg] = l[gg] * alpha + ps;
          m[gg] = mn;
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < SH::H2; ++e) acc[gg][e] = fmul2(acc[gg][e], a2);
        }
        // weighted sum of V rows
#pragma unroll
        for (int k = 0; k < SH::TB; ++k) {
          const int row = (bt * SH::TB + k) * SH::SG + grp;
          if (!full && row >= rows) continue;
#pragma unroll
          for (int c = 0; c < SH::NCH; ++c) {
            const uint4 raw =
                *reinterpret_cast<const uint4*>(vt + row * SH::ROW_BYTES + (c * SH::LPR + gl) * 16);
            const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 vf = __half22float2(h[e]);
#pragma unroll
              for (int gg = 0; gg < G; ++gg)
                acc[gg][c * 4 + e] = ffma2(make_float2(pr[k][gg], pr[k][gg]), vf, acc[gg][c * 4 + e]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
    }
    g += nb;

    // ---- merge the row groups of this warp (lanes with equal gl) ----
#pragma unroll
    for (int off = SH::LPR; off < 32; off <<= 1) {
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[gg], off);
        const float lo = __shfl_xor_sync(0xffffffffu, l[gg], off);
        const float mn = fmaxf(m[gg], mo);
        const float mu = mn == -INFINITY ? 0.f : mn;
        const float wa = fast_exp2(m[gg] - mu), wb = fast_exp2(mo - mu);
        l[gg] = l[gg] * wa + lo * wb;
        m[gg] = mn;
#pragma unroll
        for (int e = 0; e < SH::H2; ++e) {
          float2 o;
          o.x = __shfl_xor_sync(0xffffffffu, acc[gg][e].x, off);
          o.y = __shfl_xor_sync(0xffffffffu, acc[gg][e].y, off);
          acc[gg][e] = ffma2(make_float2(wb, wb), o, fmul2(acc[gg][e], make_float2(wa, wa)));
        }
      }
    }
    // ---- across warps through shared memory ----
    if (grp == 0) {
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float* dst = m_acc + (cw * G + gg) * D;
#pragma unroll
        for (int c = 0; c < SH::NCH; ++c) {
          float4* d4 = reinterpret_cast<float4*>(dst + (c * SH::LPR + gl) * 8);
          d4[0] = make_float4(acc[gg][c * 4 + 0].x, acc[gg][c * 4 + 0].y, acc[gg][c * 4 + 1].x,
                              acc[gg][c * 4 + 1].y);
          d4[1] = make_float4(acc[gg][c * 4 + 2].x, acc[gg][c * 4 + 2].y, acc[gg][c * 4 + 3].x,
                              acc[gg][c * 4 + 3].y);
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        m_ml[(cw * G + gg) * 2] = m[gg];
        m_ml[(cw * G + gg) * 2 + 1] = l[gg];
      }
    }
    consumer_sync();
    const long long rec =
        (static_cast<long long>(it.seq) * Hkv + it.kvh) * p.max_splits + it.split;
    for (int idx = ct; idx < G * D; idx += kConsumerWarps * 32) {
      const int gg = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int x = 0; x < kConsumerWarps; ++x) M = fmaxf(M, m_ml[(x * G + gg) * 2]);
      const float mu = M == -INFINITY ? 0.f : M;
      float Ls = 0.f, A = 0.f;
#pragma unroll
      for (int x = 0; x < kConsumerWarps; ++x) {
        const float wgt = fast_exp2(m_ml[(x * G + gg) * 2] - mu);
        Ls += m_ml[(x * G + gg) * 2 + 1] * wgt;
        A += m_acc[(x * G + gg) * D + d] * wgt;
      }
      if (nsplit == 1) {
        p.out[(static_cast<long long>(it.seq) * p.num_q_heads + head0 + gg) * D + d] =
            __float2half_rn(Ls > 0.f ? A / Ls : 0.f);
      } else {
        p.part_acc[rec * (G * D) + idx] = A;
        if (d == 0) {
          p.part_ml[(rec * G + gg) * 2] = M;
          p.part_ml[(rec * G + gg) * 2 + 1] = Ls;
        }
      }
    }
    if (nsplit > 1) {
      __threadfence();
      consumer_sync();
      int* cnt = p.counters + static_cast<long long>(it.seq) * Hkv + it.kvh;
      if (ct == 0) flags[1] = (atomicAdd(cnt, 1) == nsplit - 1) ? 1 : 0;
      consumer_sync();
      if (flags[1]) {
        __threadfence();
        const long long rec0 = (static_cast<long long>(it.seq) * Hkv + it.kvh) * p.max_splits;
        for (int idx = ct; idx < G * D; idx += kConsumerWarps * 32) {
          const int gg = idx / D, d = idx % D;
          float M = -INFINITY;
          for (int x = 0; x < nsplit; ++x) M = fmaxf(M, __ldcg(p.part_ml + ((rec0 + x) * G + gg) * 2));
          const float mu = M == -INFINITY ? 0.f : M;
          float Ls = 0.f, A = 0.f;
          for (int x = 0; x < nsplit; ++x) {
            const float mx = __ldcg(p.part_ml + ((rec0 + x) * G + gg) * 2);
            const float lx = __ldcg(p.part_ml + ((rec0 + x) * G + gg) * 2 + 1);
            const float wgt = fast_exp2(mx - mu);
            Ls += lx * wgt;
            A += __ldcg(p.part_acc + (rec0 + x) * (G * D) + idx) * wgt;
          }
          p.out[(static_cast<long long>(it.seq) * p.num_q_heads + head0 + gg) * D + d] =
              __float2half_rn(Ls > 0.f ? A / Ls : 0.f);
        }
        if (ct == 0) atomicExch(cnt, 0);
      }
    }
    consumer_sync();  // merge buffers and flags[1] are reused by the next item
  }
}

// --------------------------------------------------------------- host ---
int default_partition(int /*block_size*/) { return kDefaultPartitionTokens; }

struct Layout {
  size_t counters = 0, part_ml = 0, part_acc = 0, total = 0;
  int max_splits = 0;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

Layout workspace_layout(int S, int Hq, int Hkv, int D, int BS, int MB, int part_tokens) {
  Layout w;
  const int pb = part_tokens / BS;
  w.max_splits = (MB + pb - 1) / pb;
  const int G = Hq / Hkv;
  const size_t units = static_cast<size_t>(S) * Hkv * w.max_splits;
  w.counters = 0;
  w.part_ml = round256(static_cast<size_t>(S) * Hkv * 4);
  w.part_acc = w.part_ml + round256(units * G * 2 * 4);
  w.total = w.part_acc + round256(units * G * D * 4);
  return w;
}

template <int D, int BS, int G>
pa_status launch_decode(const DecodeParams& prm, const pa::DeviceInfo& dev, cudaStream_t stream) {
  using SH = Shape<D, BS, G>;
  auto kernel = paged_decode_kernel<D, BS, G>;
  const size_t smem = SH::smem_bytes(prm.num_seqs);
  if (smem > dev.smem_optin)
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_attention: %zu bytes of shared memory needed",
                    smem);
  static std::mutex mu;
  static size_t attr_set[64] = {};
  static size_t occ_smem[64] = {};
  static int occ_val[64] = {};
  int occ = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    cudaError_t e;
    if (attr_set[dev.device] < smem) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(dev.smem_optin));
      if (e != cudaSuccess) return pa::cuda_fail(e, "cudaFuncSetAttribute");
      attr_set[dev.device] = dev.smem_optin;
    }
    if (occ_smem[dev.device] != smem) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, smem);
      if (e != cudaSuccess) return pa::cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
      occ_smem[dev.device] = smem;
      occ_val[dev.device] = occ;
    }
    occ = occ_val[dev.device];
  }
  if (occ < 1) return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_attention: kernel does not fit an SM");
  const long long upper =
      static_cast<long long>(prm.num_seqs) * prm.num_kv_heads * prm.max_splits;
  long long grid = static_cast<long long>(dev.sm_count) * occ;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return pa::cuda_fail(e, "pa_decode_attention launch");
  return PA_OK;
}

template <int D, int BS>
pa_status dispatch_g(int G, const DecodeParams& prm, const pa::DeviceInfo& dev, cudaStream_t s) {
  switch (G) {
    case 1: return launch_decode<D, BS, 1>(prm, dev, s);
    case 2: return launch_decode<D, BS, 2>(prm, dev, s);
    case 4: return launch_decode<D, BS, 4>(prm, dev, s);
    case 8: return launch_decode<D, BS, 8>(prm, dev, s);
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
  if (part_tokens <= 0 || part_tokens % BS || part_tokens > 32 * BS)
    return pa::fail(PA_ERR_INVALID_ARG,
                    "partition_tokens %d must be a positive multiple of block_size <= 32 blocks",
                    part_tokens);
  if (static_cast<long long>(MB) * BS > INT32_MAX)
    return pa::fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq * block_size exceeds int32");
  return PA_OK;
}

}  // namespace

extern "C" {

size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_blocks_per_seq, int partition_tokens) {
  const int pt = partition_tokens ? partition_tokens : default_partition(block_size);
  if (check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq, pt) != PA_OK)
    return 0;
  return workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                          max_blocks_per_seq, pt)
      .total;
}

pa_status pa_decode_workspace_init(void* workspace, size_t workspace_bytes, int num_seqs,
                                   int num_kv_heads, pa_stream_t stream) {
  if (num_seqs < 0 || num_kv_heads <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "workspace_init: seqs=%d kv_heads=%d", num_seqs,
                    num_kv_heads);
  const size_t need = static_cast<size_t>(num_seqs) * num_kv_heads * 4;
  if (need == 0) return pa::ok();
  if (!workspace || workspace_bytes < need)
    return pa::fail(PA_ERR_INVALID_ARG, "workspace_init: %zu bytes < %zu", workspace_bytes, need);
  cudaError_t e = cudaMemsetAsync(workspace, 0, need, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return pa::cuda_fail(e, "workspace_init");
  return pa::ok();
}

pa_status pa_decode_attention(const pa_half* q, const pa_half* k_pool, const pa_half* v_pool,
                              const int32_t* block_table, const int32_t* seq_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks_per_seq, int num_blocks, float scale, pa_half* out,
                              void* workspace, size_t workspace_bytes, int partition_tokens,
                              pa_stream_t stream) {
  const int pt = partition_tokens ? partition_tokens : default_partition(block_size);
  if (pa_status s = check_decode_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                       max_blocks_per_seq, pt))
    return s;
  if (num_blocks <= 0 || static_cast<long long>(num_blocks) * block_size > INT32_MAX)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: num_blocks %d", num_blocks);
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: scale is not finite");
  if (num_seqs == 0) return pa::ok();
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out || !workspace)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: NULL pointer");
  if (!pa::aligned16(q) || !pa::aligned16(k_pool) || !pa::aligned16(v_pool) ||
      !pa::aligned16(out) || !pa::aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3) || (reinterpret_cast<uintptr_t>(seq_lens) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: misaligned pointer");
  const Layout lay = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                      max_blocks_per_seq, pt);
  if (workspace_bytes < lay.total)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_attention: workspace %zu < %zu bytes",
                    workspace_bytes, lay.total);
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  DecodeParams prm;
  prm.q = reinterpret_cast<const __half*>(q);
  prm.k_pool = reinterpret_cast<const __half*>(k_pool);
  prm.v_pool = reinterpret_cast<const __half*>(v_pool);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.out = reinterpret_cast<__half*>(out);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  prm.counters = reinterpret_cast<int32_t*>(ws + lay.counters);
  prm.part_ml = reinterpret_cast<float*>(ws + lay.part_ml);
  prm.part_acc = reinterpret_cast<float*>(ws + lay.part_acc);
  prm.err = pa::device_error_word();
  if (!prm.err) return PA_ERR_CUDA;
  prm.num_seqs = num_seqs;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_blocks = num_blocks;
  prm.part_blocks = pt / block_size;
  prm.max_splits = lay.max_splits;
  prm.qscale = scale * kLog2e;
  const int G = num_q_heads / num_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  pa_status st = head_dim == 64 ? dispatch_bs<64>(block_size, G, prm, dev, s)
                                : dispatch_bs<128>(block_size, G, prm, dev, s);
  return st == PA_OK ? pa::ok() : st;
}

}  // extern "C"
