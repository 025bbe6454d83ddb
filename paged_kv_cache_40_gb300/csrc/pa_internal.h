// Host-side internals shared by the libpa translation units.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "pa.h"

namespace pa {

// Record a message for pa_last_error() and return `s`.
pa_status fail(pa_status s, const char* fmt, ...);
// Clear the calling thread's message (successful call).
pa_status ok();

// Device error word of the current device (a file-scope __device__ int32
// in pa_cache.cu), resolved once per device. Returns nullptr and records a
// message on failure.
int32_t* device_error_word();

// Map a CUDA runtime error to a status with a message naming `what`.
pa_status cuda_fail(int cuda_err, const char* what);

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

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
