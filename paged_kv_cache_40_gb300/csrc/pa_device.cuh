// Device helpers shared by libpa's kernels: PTX wrappers for shared-memory
// addresses, mbarriers, bulk and tensor copies, fences, exp2 and packing; the
// bounded warp wait every pipeline uses; and the size of a partial record,
// which the attention kernel and the shared-prefix kernel both write.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_internal.h"

namespace {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // a bounded wait gives up after ~1 s
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
// Release/acquire fence at GPU scope (orders this thread's earlier and later
// memory operations around a relaxed atomic).
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two E4M3 bytes (low 16 bits of v) -> two fp16 (f16x2, byte 0 in the low
// half); exact, every E4M3 value is an fp16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t r;
  const uint16_t b = static_cast<uint16_t>(v);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(b));
  return r;
}
// Byte permute: result byte i = byte (sel >> 4i) & 7 of {b, a} (a = bytes 0..3).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// Transpose of an 8x8 matrix of 16-bit values held one row-pair per lane in
// the mma fragment layout (lane t: row t/4, columns 2(t%4), 2(t%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
// D = A * B + D, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Warp-collective bounded wait on an mbarrier phase. Every lane polls (so
// each lane itself observes the phase completion); the give-up decision is
// taken by lane 0 and broadcast, so the result is warp-uniform. Returns false
// if the phase does not complete within the time limit (the CTA is then
// flagged as aborted and PA_DEVERR_TIMEOUT recorded once) or if the CTA was
// already aborted. A warp that is not latency critical passes kSleepNs > 0 to
// sleep between polls and leave the issue slots to the warps that are.
// `limit_ns` is the time limit (about a second unless a test shortens it).
template <unsigned kSleepNs = 0>
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, int32_t* err,
                                                unsigned long long limit_ns = kWaitLimitNs) {
  const int lane = threadIdx.x & 31;
  unsigned long long t0 = 0;
  for (int iter = 0;; ++iter) {
    const bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if (kSleepNs > 0) __nanosleep(kSleepNs);
    int give_up = 0;
    if (lane == 0) {
      if (iter == 0) {
        t0 = global_ns();
      } else if (*abort_flag) {
        give_up = 1;
      } else if (global_ns() - t0 > limit_ns) {
        if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) atomicOr(err, PA_DEVERR_TIMEOUT);
        give_up = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}


// A partial record holds acc [G][D] then (max, sum) per head, padded to a
// multiple of 4 floats so every record starts on a 16-byte boundary.
__host__ __device__ constexpr int rec_floats(int G, int D) { return (G * (D + 2) + 3) / 4 * 4; }

// TMA tiled copy of box {x, y, z, w} of a 4-D tensor map into this CTA's
// shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

}  // namespace
