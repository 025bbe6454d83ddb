// Status codes, per-thread error messages and device queries for libpa.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "pa_internal.h"

namespace {
thread_local std::string g_last_error;

struct DevCache {
  std::mutex mu;
  pa::DeviceInfo info[pa::kMaxDevices];
  bool valid[pa::kMaxDevices] = {};
};
DevCache& dev_cache() {
  static DevCache c;
  return c;
}
}  // namespace

namespace pa {

pa_status fail(pa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

pa_status ok() {
  g_last_error.clear();
  return PA_OK;
}

pa_status cuda_fail(int err, const char* what) {
  cudaError_t e = static_cast<cudaError_t>(err);
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return fail(PA_ERR_UNSUPPORTED, "%s: %s (libpa is built for sm_103a only)", what,
                cudaGetErrorString(e));
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

pa_status current_device(DeviceInfo* out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (!device_slot_ok(dev))
    return fail(PA_ERR_UNSUPPORTED, "device index %d (libpa serves devices 0..%d)", dev,
                kMaxDevices - 1);
  DevCache& c = dev_cache();
  std::lock_guard<std::mutex> lock(c.mu);
  if (!c.valid[dev]) {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) ||
        (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
        (e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.smem_optin = static_cast<size_t>(v);
    c.info[dev] = d;
    c.valid[dev] = true;
  }
  *out = c.info[dev];
  if (out->cc_major != 10 || out->cc_minor != 3)
    return fail(PA_ERR_UNSUPPORTED, "device %d is sm_%d%d; libpa is built for sm_103a only",
                dev, out->cc_major, out->cc_minor);
  return PA_OK;
}

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace pa

extern "C" {

uint64_t pa_kernel_launches(void) { return pa::g_launches.load(std::memory_order_relaxed); }

const char* pa_last_error(void) { return g_last_error.c_str(); }

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS";
    case PA_ERR_BAD_BLOCK_ID: return "PA_ERR_BAD_BLOCK_ID";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
  }
  return "PA_ERR_UNKNOWN";
}

int pa_version(void) { return 300; }

}  // extern "C"
