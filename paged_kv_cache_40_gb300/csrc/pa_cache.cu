// KV-cache writes: per-token append through a slot mapping, and whole-block
// copy-on-write duplication. Both are pure bit copies streamed with 16-byte
// vector loads/stores; a block is block_size consecutive rows of
// num_kv_heads*head_dim values, and consecutive blocks of a pool sit a block
// stride apart (the dense stride for two separate pools, twice a block for
// the one-pool record layout of the layout sketch, where each record holds a
// block's K rows and then its V rows: Document 04, §2 Core Concept).
//
// Append: the cache grows by one token per decode step ("Phase 7 · Document
// 04 — PagedAttention", §2 primer); the block manager picks the slot (§2 Core
// Concept, on-demand allocation). Copy: copy-on-write of a shared block (§2
// "block sharing", §3 Mental Model; lux-666 notes "PagedAttention", prefix
// sharing section).
//
// fp8 cache (Document 04, §11: `--kv-cache-dtype fp8`, KV quantization to fit
// more sequences): the append quantizes each fp16 value to an OCP E4M3 byte,
// code = e4m3(fp32(x) / scale[head]) with the division in IEEE fp32 and the
// conversion rounding to nearest even and saturating at +-448; the block copy
// is the same bit copy over one-byte elements.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <utility>

#include "pa_internal.h"

// Device error word: bits PA_DEVERR_* set by any libpa kernel that skipped
// an out-of-range access. Read and cleared by pa_device_error().
__device__ int32_t g_pa_device_error = 0;

namespace {

// Launch `kernel` on `stream` as a programmatic dependent of the kernel
// ahead of it: its CTAs may be scheduled while that one finishes, and wait
// (griddepcontrol.wait) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, int threads, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(threads);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

constexpr int kAppendThreads = 128;
constexpr int kCopyThreads = 256;
constexpr int kCopyVecsPerThread = 4;

// One CTA per appended token: copy its K row and V row (row_vecs 16-byte
// vectors each) into pool row `slot`.
__global__ void __launch_bounds__(kAppendThreads)
append_kv_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                 uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                 const int32_t* __restrict__ slots, int row_vecs, int block_size,
                 int64_t block_vecs, int64_t num_slots, int32_t* __restrict__ err) {
  // A decode launched right after this kernel may start its prologue now; it
  // waits for this grid to finish before it reads the pool. This kernel is
  // itself launched as a programmatic dependent (of the copy-on-write copies,
  // say): it reads nothing before the kernel ahead of it has completed.
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x;
  const int32_t slot = __ldg(slots + t);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0) atomicOr(err, PA_DEVERR_BAD_SLOT);
    return;
  }
  const uint4* ks = k_new + static_cast<int64_t>(t) * row_vecs;
  const uint4* vs = v_new + static_cast<int64_t>(t) * row_vecs;
  const int64_t row = (slot / block_size) * block_vecs +
                      static_cast<int64_t>(slot % block_size) * row_vecs;
  uint4* kd = k_pool + row;
  uint4* vd = v_pool + row;
  for (int i = threadIdx.x; i < row_vecs; i += kAppendThreads) {
    const uint4 a = __ldg(ks + i);
    const uint4 b = __ldg(vs + i);
    kd[i] = a;
    vd[i] = b;
  }
}

// Two fp32 values -> two E4M3 bytes (lo in the low byte), round to nearest
// even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One CTA per appended token: quantize its K row and V row (Hkv*D fp16 each)
// to E4M3 and store them in pool row `slot`. Each thread takes 8 values (one
// 16-byte load, one 8-byte store) of one head.
__global__ void __launch_bounds__(kAppendThreads)
append_kv_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint2* __restrict__ k_pool, uint2* __restrict__ v_pool,
                     const int32_t* __restrict__ slots, const float* __restrict__ k_scale,
                     const float* __restrict__ v_scale, int row_vecs, int head_vecs,
                     int block_size, int64_t block_vecs, int64_t num_slots,
                     int32_t* __restrict__ err) {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x;
  const int32_t slot = __ldg(slots + t);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0) atomicOr(err, PA_DEVERR_BAD_SLOT);
    return;
  }
  const uint4* ks = k_new + static_cast<int64_t>(t) * row_vecs;
  const uint4* vs = v_new + static_cast<int64_t>(t) * row_vecs;
  const int64_t row = (slot / block_size) * block_vecs +
                      static_cast<int64_t>(slot % block_size) * row_vecs;
  uint2* kd = k_pool + row;
  uint2* vd = v_pool + row;
  for (int i = threadIdx.x; i < row_vecs; i += kAppendThreads) {
    const int h = i / head_vecs;
    const float sk = __ldg(k_scale + h), sv = __ldg(v_scale + h);
    const uint4 a = __ldg(ks + i);
    const uint4 b = __ldg(vs + i);
    const __half2* ah = reinterpret_cast<const __half2*>(&a);
    const __half2* bh = reinterpret_cast<const __half2*>(&b);
    uint32_t ko[2] = {0, 0}, vo[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = __half22float2(ah[j]);
      const float2 y = __half22float2(bh[j]);
      const uint32_t kq = f32x2_to_e4m3x2(__fdiv_rn(x.x, sk), __fdiv_rn(x.y, sk));
      const uint32_t vq = f32x2_to_e4m3x2(__fdiv_rn(y.x, sv), __fdiv_rn(y.y, sv));
      ko[j >> 1] |= kq << (16 * (j & 1));
      vo[j >> 1] |= vq << (16 * (j & 1));
    }
    kd[i] = make_uint2(ko[0], ko[1]);
    vd[i] = make_uint2(vo[0], vo[1]);
  }
}

// Grid (pairs, slices): each CTA copies a slice of one block of the source
// pools into a block of the destination pools (the same pools for
// copy-on-write; the device pools and a host pool for swapping). Blocks are
// block_vecs long and sit src_stride / dst_stride vectors apart; with no V
// pools (src_v == dst_v == nullptr) only the K side is copied.
__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                   uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                   const int32_t* __restrict__ pairs, int64_t block_vecs, int64_t src_stride,
                   int64_t dst_stride, int src_blocks, int dst_blocks,
                   int32_t* __restrict__ err) {
  // the append that follows may launch now; it waits for this grid before it
  // writes. Launched as a programmatic dependent itself, this kernel touches
  // nothing before the kernel ahead of it has completed.
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int p = blockIdx.x;
  const int32_t src = __ldg(pairs + 2 * p);
  const int32_t dst = __ldg(pairs + 2 * p + 1);
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(err, PA_DEVERR_BAD_BLOCK);
    return;
  }
  const int64_t slice = static_cast<int64_t>(kCopyThreads) * kCopyVecsPerThread;
  const int64_t lo = blockIdx.y * slice;
  const int64_t hi = lo + slice < block_vecs ? lo + slice : block_vecs;
  const bool two = src_v != nullptr;
  const uint4* ks = src_k + src * src_stride;
  const uint4* vs = two ? src_v + src * src_stride : nullptr;
  uint4* kd = dst_k + dst * dst_stride;
  uint4* vd = two ? dst_v + dst * dst_stride : nullptr;
  uint4 kb[kCopyVecsPerThread], vb[kCopyVecsPerThread];
#pragma unroll
  for (int j = 0; j < kCopyVecsPerThread; ++j) {
    const int64_t i = lo + threadIdx.x + j * kCopyThreads;
    if (i < hi) {
      kb[j] = ks[i];
      if (two) vb[j] = vs[i];
    }
  }
#pragma unroll
  for (int j = 0; j < kCopyVecsPerThread; ++j) {
    const int64_t i = lo + threadIdx.x + j * kCopyThreads;
    if (i < hi) {
      kd[i] = kb[j];
      if (two) vd[i] = vb[j];
    }
  }
}

pa_status check_pool_shape(const char* fn, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks) {
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "%s: kv_heads=%d head_dim=%d block_size=%d blocks=%d",
                    fn, num_kv_heads, head_dim, block_size, num_blocks);
  if (head_dim % 8)
    return pa::fail(PA_ERR_UNSUPPORTED, "%s: head_dim %d is not a multiple of 8", fn, head_dim);
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
    return pa::fail(PA_ERR_INVALID_ARG, "%s: pool slots exceed int32", fn);
  return PA_OK;
}

// Block stride (values) of the K and V pools a writing call gets, checked:
// a valid stride and K blocks that do not overlap V blocks.
pa_status writer_stride(const char* fn, const void* k_pool, const void* v_pool, int num_kv_heads,
                        int head_dim, int block_size, int num_blocks, int64_t stride, int esz,
                        int64_t* out) {
  const int64_t dense = static_cast<int64_t>(block_size) * num_kv_heads * head_dim;
  if (pa_status s = pa::resolve_block_stride(fn, stride, dense, esz, out)) return s;
  return pa::check_pools_disjoint(fn, k_pool, v_pool, num_blocks, *out * esz, dense * esz);
}

}  // namespace

namespace pa {

pa_status resolve_block_stride(const char* fn, int64_t stride, int64_t dense, int esz,
                               int64_t* out) {
  if (stride == 0) {
    *out = dense;
    return PA_OK;
  }
  if (stride < dense || (stride * esz) % 16 != 0 || stride > (int64_t{1} << 40) / esz)
    return fail(PA_ERR_INVALID_ARG,
                "%s: pool_block_stride %lld values (a block holds %lld; the stride must be at "
                "least that and a multiple of 16 bytes)",
                fn, static_cast<long long>(stride), static_cast<long long>(dense));
  *out = stride;
  return PA_OK;
}

pa_status check_pools_disjoint(const char* fn, const void* k, const void* v, int num_blocks,
                               int64_t stride_bytes, int64_t block_bytes) {
  const int64_t span = (static_cast<int64_t>(num_blocks) - 1) * stride_bytes + block_bytes;
  const int64_t kb = static_cast<int64_t>(reinterpret_cast<uintptr_t>(k));
  const int64_t vb = static_cast<int64_t>(reinterpret_cast<uintptr_t>(v));
  const int64_t delta = vb - kb;
  if (delta >= span || -delta >= span) return PA_OK;  // the pools' extents do not meet
  // Interleaved extents: every V block must fall in a gap between K blocks.
  const int64_t r = ((delta % stride_bytes) + stride_bytes) % stride_bytes;
  if (r >= block_bytes && r <= stride_bytes - block_bytes) return PA_OK;
  return fail(PA_ERR_INVALID_ARG, "%s: K and V pool blocks overlap (v - k = %lld bytes, block "
              "%lld bytes, stride %lld bytes)", fn, static_cast<long long>(delta),
              static_cast<long long>(block_bytes), static_cast<long long>(stride_bytes));
}

int32_t* device_error_word() {
  static std::mutex mu;
  static int32_t* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || !device_slot_ok(dev)) {
    fail(PA_ERR_CUDA, "device_error_word: no current device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_pa_device_error);
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaGetSymbolAddress(device error word)");
      return nullptr;
    }
    addr[dev] = static_cast<int32_t*>(p);
  }
  return addr[dev];
}

}  // namespace pa

extern "C" {

pa_status pa_device_error(pa_stream_t stream, int32_t* flags) {
  if (!flags) return pa::fail(PA_ERR_INVALID_ARG, "pa_device_error: flags is NULL");
  *flags = 0;
  int32_t* word = pa::device_error_word();
  if (!word) return PA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, word, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return pa::cuda_fail(e, "pa_device_error");
  *flags = host;
  if (host & PA_DEVERR_TIMEOUT)
    return pa::fail(PA_ERR_TIMEOUT, "a device pipeline wait hit its time limit (flags 0x%x)", host);
  if (host)
    return pa::fail(PA_ERR_BAD_BLOCK_ID,
                    "device skipped out-of-range accesses (flags 0x%x: 1=block id, 2=slot, "
                    "4=length)", host);
  return pa::ok();
}

pa_status pa_append_kv(const pa_half* k_new, const pa_half* v_new, pa_half* k_pool,
                       pa_half* v_pool, const int32_t* slot_mapping, int num_tokens,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       int64_t pool_block_stride, pa_stream_t stream) {
  if (pa_status s = check_pool_shape("pa_append_kv", num_kv_heads, head_dim, block_size,
                                     num_blocks))
    return s;
  if (num_tokens < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_append_kv: num_tokens < 0");
  if (num_tokens == 0) return pa::ok();
  if (!k_new || !v_new || !k_pool || !v_pool || !slot_mapping)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_append_kv: NULL pointer");
  if (!pa::aligned16(k_new) || !pa::aligned16(v_new) || !pa::aligned16(k_pool) ||
      !pa::aligned16(v_pool) || (reinterpret_cast<uintptr_t>(slot_mapping) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_append_kv: misaligned pointer");
  int64_t stride = 0;
  if (pa_status s = writer_stride("pa_append_kv", k_pool, v_pool, num_kv_heads, head_dim,
                                  block_size, num_blocks, pool_block_stride, 2, &stride))
    return s;
  if (pa_status s = pa::device_only("pa_append_kv(k_pool)", k_pool)) return s;
  if (pa_status s = pa::device_in("pa_append_kv(k_new)", k_new)) return s;
  if (pa_status s = pa::device_in("pa_append_kv(v_new)", v_new)) return s;
  if (pa_status s = pa::device_in("pa_append_kv(slot_mapping)", slot_mapping)) return s;
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  int32_t* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  {
    // Same shared-memory carveout as the attention kernel that usually
    // follows, so its CTAs can start on SMs this kernel still occupies.
    static std::mutex mu;
    static bool set[pa::kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev.device]) {
      cudaError_t e = cudaFuncSetAttribute(append_kv_kernel,
                                           cudaFuncAttributePreferredSharedMemoryCarveout,
                                           cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return pa::cuda_fail(e, "cudaFuncSetAttribute(append)");
      set[dev.device] = true;
    }
  }
  const int row_vecs = num_kv_heads * head_dim / 8;
  cudaError_t e = launch_dependent(
      append_kv_kernel, dim3(num_tokens), kAppendThreads, static_cast<cudaStream_t>(stream),
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(v_pool), slot_mapping,
      row_vecs, block_size, stride / 8, static_cast<int64_t>(num_blocks) * block_size, err);
  if (e != cudaSuccess) return pa::cuda_fail(e, "pa_append_kv launch");
  pa::count_launch();
  return pa::ok();
}

pa_status pa_copy_blocks(pa_half* k_pool, pa_half* v_pool, const int32_t* pairs,
                         int num_pairs, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int64_t pool_block_stride, pa_stream_t stream) {
  if (pa_status s = check_pool_shape("pa_copy_blocks", num_kv_heads, head_dim, block_size,
                                     num_blocks))
    return s;
  if (num_pairs < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: num_pairs < 0");
  if (num_pairs == 0) return pa::ok();
  if (!k_pool || !v_pool || !pairs)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: NULL pointer");
  if (!pa::aligned16(k_pool) || !pa::aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(pairs) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: misaligned pointer");
  int64_t stride = 0;
  if (pa_status s = writer_stride("pa_copy_blocks", k_pool, v_pool, num_kv_heads, head_dim,
                                  block_size, num_blocks, pool_block_stride, 2, &stride))
    return s;
  if (pa_status s = pa::device_only("pa_copy_blocks(k_pool)", k_pool)) return s;
  if (pa_status s = pa::device_in("pa_copy_blocks(pairs)", pairs)) return s;
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  int32_t* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  const int64_t block_vecs = static_cast<int64_t>(block_size) * num_kv_heads * head_dim / 8;
  const int64_t slice = static_cast<int64_t>(kCopyThreads) * kCopyVecsPerThread;
  const int64_t slices = (block_vecs + slice - 1) / slice;
  if (slices > 65535) return pa::fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks: block too large");
  dim3 grid(num_pairs, static_cast<unsigned>(slices));
  cudaError_t e = launch_dependent(
      copy_blocks_kernel, grid, kCopyThreads, static_cast<cudaStream_t>(stream),
      reinterpret_cast<const uint4*>(k_pool), reinterpret_cast<const uint4*>(v_pool),
      reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(v_pool), pairs, block_vecs,
      stride / 8, stride / 8, num_blocks, num_blocks, err);
  if (e != cudaSuccess) return pa::cuda_fail(e, "pa_copy_blocks launch");
  pa::count_launch();
  return pa::ok();
}

pa_status pa_append_kv_fp8(const pa_half* k_new, const pa_half* v_new, uint8_t* k_pool,
                           uint8_t* v_pool, const int32_t* slot_mapping, const float* k_scale,
                           const float* v_scale, int num_tokens, int num_kv_heads, int head_dim,
                           int block_size, int num_blocks, int64_t pool_block_stride,
                           pa_stream_t stream) {
  if (pa_status s = check_pool_shape("pa_append_kv_fp8", num_kv_heads, head_dim, block_size,
                                     num_blocks))
    return s;
  if (num_tokens < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_append_kv_fp8: num_tokens < 0");
  if (num_tokens == 0) return pa::ok();
  if (!k_new || !v_new || !k_pool || !v_pool || !slot_mapping || !k_scale || !v_scale)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_append_kv_fp8: NULL pointer");
  if (!pa::aligned16(k_new) || !pa::aligned16(v_new) || !pa::aligned16(k_pool) ||
      !pa::aligned16(v_pool) || (reinterpret_cast<uintptr_t>(slot_mapping) & 3) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3) || (reinterpret_cast<uintptr_t>(v_scale) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_append_kv_fp8: misaligned pointer");
  int64_t stride = 0;
  if (pa_status s = writer_stride("pa_append_kv_fp8", k_pool, v_pool, num_kv_heads, head_dim,
                                  block_size, num_blocks, pool_block_stride, 1, &stride))
    return s;
  if (pa_status s = pa::device_only("pa_append_kv_fp8(k_pool)", k_pool)) return s;
  if (pa_status s = pa::device_in("pa_append_kv_fp8(k_new)", k_new)) return s;
  if (pa_status s = pa::device_in("pa_append_kv_fp8(v_new)", v_new)) return s;
  if (pa_status s = pa::device_in("pa_append_kv_fp8(slot_mapping)", slot_mapping)) return s;
  if (pa_status s = pa::device_in("pa_append_kv_fp8(k_scale)", k_scale)) return s;
  if (pa_status s = pa::device_in("pa_append_kv_fp8(v_scale)", v_scale)) return s;
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  int32_t* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  {
    static std::mutex mu;
    static bool set[pa::kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev.device]) {
      cudaError_t e = cudaFuncSetAttribute(append_kv_fp8_kernel,
                                           cudaFuncAttributePreferredSharedMemoryCarveout,
                                           cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return pa::cuda_fail(e, "cudaFuncSetAttribute(append fp8)");
      set[dev.device] = true;
    }
  }
  const int row_vecs = num_kv_heads * head_dim / 8;
  cudaError_t e = launch_dependent(
      append_kv_fp8_kernel, dim3(num_tokens), kAppendThreads, static_cast<cudaStream_t>(stream),
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      reinterpret_cast<uint2*>(k_pool), reinterpret_cast<uint2*>(v_pool), slot_mapping, k_scale,
      v_scale, row_vecs, head_dim / 8, block_size, stride / 8,
      static_cast<int64_t>(num_blocks) * block_size, err);
  if (e != cudaSuccess) return pa::cuda_fail(e, "pa_append_kv_fp8 launch");
  pa::count_launch();
  return pa::ok();
}

pa_status pa_copy_blocks_fp8(uint8_t* k_pool, uint8_t* v_pool, const int32_t* pairs,
                             int num_pairs, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, int64_t pool_block_stride, pa_stream_t stream) {
  if (pa_status s = check_pool_shape("pa_copy_blocks_fp8", num_kv_heads, head_dim, block_size,
                                     num_blocks))
    return s;
  if (head_dim % 16)
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks_fp8: head_dim %d not a multiple of 16",
                    head_dim);
  if (num_pairs < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks_fp8: num_pairs < 0");
  if (num_pairs == 0) return pa::ok();
  if (!k_pool || !v_pool || !pairs)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks_fp8: NULL pointer");
  if (!pa::aligned16(k_pool) || !pa::aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(pairs) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks_fp8: misaligned pointer");
  int64_t stride = 0;
  if (pa_status s = writer_stride("pa_copy_blocks_fp8", k_pool, v_pool, num_kv_heads, head_dim,
                                  block_size, num_blocks, pool_block_stride, 1, &stride))
    return s;
  if (pa_status s = pa::device_only("pa_copy_blocks_fp8(k_pool)", k_pool)) return s;
  if (pa_status s = pa::device_in("pa_copy_blocks_fp8(pairs)", pairs)) return s;
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  int32_t* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  const int64_t block_vecs = static_cast<int64_t>(block_size) * num_kv_heads * head_dim / 16;
  const int64_t slice = static_cast<int64_t>(kCopyThreads) * kCopyVecsPerThread;
  const int64_t slices = (block_vecs + slice - 1) / slice;
  if (slices > 65535) return pa::fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks_fp8: block too large");
  dim3 grid(num_pairs, static_cast<unsigned>(slices));
  cudaError_t e = launch_dependent(
      copy_blocks_kernel, grid, kCopyThreads, static_cast<cudaStream_t>(stream),
      reinterpret_cast<const uint4*>(k_pool), reinterpret_cast<const uint4*>(v_pool),
      reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(v_pool), pairs, block_vecs,
      stride / 16, stride / 16, num_blocks, num_blocks, err);
  if (e != cudaSuccess) return pa::cuda_fail(e, "pa_copy_blocks_fp8 launch");
  pa::count_launch();
  return pa::ok();
}

}  // extern "C"

namespace pa {

pa_status device_view(const char* fn, const void* p, void** out) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) return pa::cuda_fail(e, fn);
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *out = const_cast<void*>(p);
    return PA_OK;
  }
  if (at.type == cudaMemoryTypeHost) {
    void* d = nullptr;
    e = cudaHostGetDevicePointer(&d, const_cast<void*>(p), 0);
    if (e != cudaSuccess) return pa::cuda_fail(e, fn);
    *out = d;
    return PA_OK;
  }
  return pa::fail(PA_ERR_INVALID_ARG, "%s: host memory must be pinned (page-locked)", fn);
}

pa_status device_only(const char* fn, const void* p) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) return pa::cuda_fail(e, fn);
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return PA_OK;
  return pa::fail(PA_ERR_INVALID_ARG, "%s: must be device memory", fn);
}

}  // namespace pa

extern "C" {

pa_status pa_swap_blocks(const void* src_k, const void* src_v, int src_blocks,
                         int64_t src_block_stride, void* dst_k, void* dst_v, int dst_blocks,
                         int64_t dst_block_stride, const int32_t* pairs, int num_pairs,
                         int block_bytes, pa_stream_t stream) {
  if (num_pairs < 0 || src_blocks <= 0 || dst_blocks <= 0 || block_bytes <= 0 ||
      block_bytes % 16)
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_swap_blocks: pairs=%d src_blocks=%d dst_blocks=%d block_bytes=%d",
                    num_pairs, src_blocks, dst_blocks, block_bytes);
  int64_t src_stride = 0, dst_stride = 0;
  if (pa_status s = pa::resolve_block_stride("pa_swap_blocks(src)", src_block_stride,
                                             block_bytes, 1, &src_stride))
    return s;
  if (pa_status s = pa::resolve_block_stride("pa_swap_blocks(dst)", dst_block_stride,
                                             block_bytes, 1, &dst_stride))
    return s;
  if (num_pairs == 0) return pa::ok();
  const bool two = src_v != nullptr;
  if (!src_k || !dst_k || !pairs || two != (dst_v != nullptr))
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_swap_blocks: NULL pointer (src_v and dst_v are both set or both NULL)");
  if (!pa::aligned16(src_k) || !pa::aligned16(src_v) || !pa::aligned16(dst_k) ||
      !pa::aligned16(dst_v) || (reinterpret_cast<uintptr_t>(pairs) & 3))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: misaligned pointer");
  if (two) {
    if (pa_status s = pa::check_pools_disjoint("pa_swap_blocks(dst)", dst_k, dst_v, dst_blocks,
                                               dst_stride, block_bytes))
      return s;
  }
  pa::DeviceInfo dev;
  if (pa_status s = pa::current_device(&dev)) return s;
  void *sk = nullptr, *sv = nullptr, *dk = nullptr, *dv = nullptr, *pp = nullptr;
  if (pa_status s = pa::device_view("pa_swap_blocks(src_k)", src_k, &sk)) return s;
  if (pa_status s = pa::device_view("pa_swap_blocks(dst_k)", dst_k, &dk)) return s;
  if (two) {
    if (pa_status s = pa::device_view("pa_swap_blocks(src_v)", src_v, &sv)) return s;
    if (pa_status s = pa::device_view("pa_swap_blocks(dst_v)", dst_v, &dv)) return s;
  }
  if (pa_status s = pa::device_view("pa_swap_blocks(pairs)", pairs, &pp)) return s;
  int32_t* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  const int64_t block_vecs = block_bytes / 16;
  const int64_t slice = static_cast<int64_t>(kCopyThreads) * kCopyVecsPerThread;
  const int64_t slices = (block_vecs + slice - 1) / slice;
  if (slices > 65535) return pa::fail(PA_ERR_UNSUPPORTED, "pa_swap_blocks: block too large");
  dim3 grid(num_pairs, static_cast<unsigned>(slices));
  copy_blocks_kernel<<<grid, kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(sk), static_cast<const uint4*>(sv), static_cast<uint4*>(dk),
      static_cast<uint4*>(dv), static_cast<const int32_t*>(pp), block_vecs, src_stride / 16,
      dst_stride / 16, src_blocks, dst_blocks, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return pa::cuda_fail(e, "pa_swap_blocks launch");
  pa::count_launch();
  return pa::ok();
}

}  // extern "C"
