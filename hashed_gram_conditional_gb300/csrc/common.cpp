// Error reporting, device checks and version queries of libengram.
#include <cuda_runtime.h>

#include <atomic>
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

namespace {
// Process-wide kernel options, one relaxed atomic per field.
std::atomic<int32_t> g_opt_projection_cta{0}, g_opt_gather_copy{0}, g_opt_fp8_pair{0}, g_opt_fp8_fused{0},
    g_opt_plain_launch{0};
}  // namespace

engram_kernel_options kernel_options() {
  engram_kernel_options o;
  o.projection_cta = g_opt_projection_cta.load(std::memory_order_relaxed);
  o.gather_copy = g_opt_gather_copy.load(std::memory_order_relaxed);
  o.fp8_pair = g_opt_fp8_pair.load(std::memory_order_relaxed);
  o.fp8_fused = g_opt_fp8_fused.load(std::memory_order_relaxed);
  o.plain_launch = g_opt_plain_launch.load(std::memory_order_relaxed);
  return o;
}

}  // namespace engram

extern "C" {

int engram_set_kernel_options(const engram_kernel_options* opts) {
  using namespace engram;
  if (opts == nullptr) return fail(ENGRAM_E_INVALID, "null kernel options");
  if (opts->projection_cta < 0 || opts->projection_cta > 2 || opts->gather_copy < 0 || opts->gather_copy > 1 ||
      opts->fp8_pair < 0 || opts->fp8_pair > 1 || opts->fp8_fused < 0 || opts->fp8_fused > 1 ||
      opts->plain_launch < 0 || opts->plain_launch > 1)
    return fail(ENGRAM_E_INVALID, "kernel option out of range");
  g_opt_projection_cta.store(opts->projection_cta, std::memory_order_relaxed);
  g_opt_gather_copy.store(opts->gather_copy, std::memory_order_relaxed);
  g_opt_fp8_pair.store(opts->fp8_pair, std::memory_order_relaxed);
  g_opt_fp8_fused.store(opts->fp8_fused, std::memory_order_relaxed);
  g_opt_plain_launch.store(opts->plain_launch, std::memory_order_relaxed);
  return ENGRAM_OK;
}

int engram_get_kernel_options(engram_kernel_options* out) {
  if (out == nullptr) return engram::fail(ENGRAM_E_INVALID, "null kernel options");
  *out = engram::kernel_options();
  return ENGRAM_OK;
}


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
