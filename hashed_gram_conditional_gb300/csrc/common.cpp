// Error reporting, device checks and version queries of libengram.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "engram_internal.h"

namespace engram {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int check_device(int* sm_count) {
  static std::mutex mu;
  static int cached_sm[64] = {0};
  static int cached_ok[64] = {0};  // 0 unknown, 1 ok, -1 wrong arch
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (dev < 0 || dev >= 64) return fail(ENGRAM_E_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (cached_ok[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail(ENGRAM_E_CUDA, "cudaDeviceGetAttribute failed on device %d", dev);
    cached_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    cached_sm[dev] = sms;
    if (cached_ok[dev] < 0)
      set_error("libengram is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
  }
  if (cached_ok[dev] < 0) return ENGRAM_E_DEVICE;
  if (sm_count) *sm_count = cached_sm[dev];
  return ENGRAM_OK;
}

int check_launch(const char* what) {
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "%s: %s", what, cudaGetErrorString(err));
  return ENGRAM_OK;
}

}  // namespace engram

extern "C" {

const char* engram_last_error(void) { return engram::g_last_error.c_str(); }

const char* engram_status_string(int code) {
  switch (code) {
    case ENGRAM_OK: return "ENGRAM_OK";
    case ENGRAM_E_INVALID: return "ENGRAM_E_INVALID";
    case ENGRAM_E_VOCAB: return "ENGRAM_E_VOCAB";
    case ENGRAM_E_SHAPE: return "ENGRAM_E_SHAPE";
    case ENGRAM_E_ALIGN: return "ENGRAM_E_ALIGN";
    case ENGRAM_E_RANGE: return "ENGRAM_E_RANGE";
    case ENGRAM_E_CUDA: return "ENGRAM_E_CUDA";
    case ENGRAM_E_DEVICE: return "ENGRAM_E_DEVICE";
    default: return "ENGRAM_E_UNKNOWN";
  }
}

int engram_abi_version(void) { return ENGRAM_ABI_VERSION; }

size_t engram_layout_params_size(void) { return sizeof(engram_layout_params); }
size_t engram_layout_size(void) { return sizeof(engram_layout); }

}  // extern "C"
