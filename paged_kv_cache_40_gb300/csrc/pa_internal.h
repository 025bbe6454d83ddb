// Host-side internals shared by the libpa translation units.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "pa.h"

namespace pa {

// Devices libpa keeps per-device state for (tables indexed by the device
// ordinal); current_device() refuses ordinals outside [0, kMaxDevices).
constexpr int kMaxDevices = 64;

// True for an ordinal the per-device tables can index.
inline bool device_slot_ok(int device) { return device >= 0 && device < kMaxDevices; }

// Record a message for pa_last_error() and return `s`.
pa_status fail(pa_status s, const char* fmt, ...);
// Clear the calling thread's message (successful call).
pa_status ok();

// Device error word of the current device (a file-scope __device__ int32
// in pa_cache.cu), resolved once per device. Returns nullptr and records a
// message on failure.
int32_t* device_error_word();

// Count one kernel launch the library enqueued (pa_kernel_launches).
void count_launch();

// Map a CUDA runtime error to a status with a message naming `what`.
pa_status cuda_fail(int cuda_err, const char* what);

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Block stride of a pool in values: 0 selects the dense stride `dense`
// (block_size*num_kv_heads*head_dim); otherwise the stride must be at least
// `dense` and a multiple of 16 bytes (`esz` bytes per value). Writes the
// stride in values to *out, or records a message naming `fn` and returns
// PA_ERR_INVALID_ARG.
pa_status resolve_block_stride(const char* fn, int64_t stride, int64_t dense, int esz,
                               int64_t* out);

// For calls that write both pools: blocks of `block_bytes` at k + b*stride
// and v + b*stride (b < num_blocks, stride in bytes) must not overlap between
// the two pools. Records a message naming `fn` and returns PA_ERR_INVALID_ARG
// when they do.
pa_status check_pools_disjoint(const char* fn, const void* k, const void* v, int num_blocks,
                               int64_t stride_bytes, int64_t block_bytes);

// A pointer the device can dereference: device (or managed) memory as it is,
// pinned host memory through its device mapping; pageable host memory is
// refused (PA_ERR_INVALID_ARG, message naming `fn`).
pa_status device_view(const char* fn, const void* p, void** out);

// device_view for a pointer the call reads or writes in place (NULL stays
// NULL); the const-ness of the caller's pointer is kept.
template <typename T>
pa_status device_in(const char* fn, T*& p) {
  if (!p) return PA_OK;
  void* d = nullptr;
  if (pa_status s = device_view(fn, p, &d)) return s;
  p = static_cast<T*>(d);
  return PA_OK;
}

// Memory the kernels reach through TMA or hold across calls (pools,
// workspaces) must be device memory: PA_ERR_INVALID_ARG otherwise.
pa_status device_only(const char* fn, const void* p);

// The block manager's block size and pool size (for the step driver).
int alloc_block_size(const pa_allocator* a);
int alloc_num_blocks(const pa_allocator* a);

// Properties of the current device used for launch shaping.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
};
// Cached per device; returns non-OK (with message) when no device is usable.
pa_status current_device(DeviceInfo* out);

}  // namespace pa
