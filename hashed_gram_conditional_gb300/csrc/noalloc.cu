// Projection + gate/residual stage without any device allocation.
//
// engram_project and engram_gate_add hand each other two intermediate
// buffers (the gate's partial sums and the bf16 value v), which the caller
// normally allocates.  Some callers cannot allocate device memory at the
// point where they run this stage: for example a serving engine that has
// reserved the whole of HBM up front for its own pools (KV cache, weights)
// and forbids cudaMalloc on its hot path, or a plugin that runs inside a
// host framework whose allocator it does not own.  This entry point serves
// them: its intermediates live in one file-scope device array of fixed size,
// so the caller passes only its inputs and outputs.
//
// The array (kScratchBytes, 8 MiB) is part of the library image: every GPU on
// which the library is loaded holds it until the process exits.  All calls
// share it, so calls that overlap on the GPU (on different streams, or from
// different threads without ordering) race on it.  Each call writes every
// scratch element it later reads, so nothing needs clearing between calls.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "engram_internal.h"

namespace engram {
namespace {

constexpr size_t kScratchBytes = ENGRAM_STAGE_STATIC_SCRATCH_BYTES;  // 8 MiB
constexpr size_t kAlign = 256;

// Host code must not use this name as a device address: it is a host-side
// shadow symbol.  The device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_stage_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Device address of g_stage_scratch on the current device, looked up once per
// device (with that device current) on the first call made there.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (dev < 0 || dev >= kMaxDevices) return fail(ENGRAM_E_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_stage_scratch);
    if (err != cudaSuccess || p == nullptr)
      return fail(ENGRAM_E_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(err));
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return ENGRAM_OK;
}

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" int engram_project_gate_add_noalloc(const uint16_t* e_d, int64_t n_tokens, int64_t K,
                                               const uint16_t* wkv_packed_d, int32_t hidden, int32_t hc,
                                               uint16_t* h_d, const float* q_w_d, const float* k_w_d,
                                               const uint8_t* mask_d, float eps, float clamp,
                                               float score_scale, float* gate_out_d, int32_t* status_d,
                                               void* stream) {
  if (n_tokens < 0) return fail(ENGRAM_E_INVALID, "n_tokens < 0");
  if (hidden < 256 || hidden % 256 != 0 || hc < 1 || hc > 8)
    return fail(ENGRAM_E_SHAPE, "hidden %d must be a multiple of 256 and hc %d in [1, 8]", hidden, hc);
  if (n_tokens == 0) return ENGRAM_OK;
  const size_t partials = engram_project_partials_bytes(n_tokens, hidden, hc);
  const size_t v_bytes = static_cast<size_t>(n_tokens) * hidden * 2;
  const size_t need = round_up(partials) + v_bytes;
  if (need > kScratchBytes) {
    const size_t per_token = engram_project_partials_bytes(1, hidden, hc) + static_cast<size_t>(hidden) * 2;
    return fail(ENGRAM_E_RANGE,
                "%lld tokens need %zu bytes of stage scratch; the static scratch holds %zu bytes "
                "(about %zu tokens at hidden %d, hc %d)",
                (long long)n_tokens, need, kScratchBytes, (kScratchBytes - kAlign) / per_token, hidden, hc);
  }
  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc) return rc;
  float* partials_d = static_cast<float*>(base);
  uint16_t* v_d = reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(base) + round_up(partials));
  rc = engram_project(e_d, n_tokens, K, wkv_packed_d, hidden, hc, h_d, q_w_d, k_w_d, partials_d, v_d, status_d,
                      stream);
  if (rc) return rc;
  return engram_gate_add(partials_d, v_d, h_d, mask_d, n_tokens, hidden, hc, eps, clamp, score_scale, gate_out_d,
                         stream);
}
