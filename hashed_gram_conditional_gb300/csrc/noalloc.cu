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
#include <cuda.h>
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
unsigned long long g_ctx_id[kMaxDevices] = {0};

// Driver calls reached through the runtime's entry-point query, so the
// library needs no link against libcuda.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

int driver_fn(const char* name, void** fn) {
  cudaDriverEntryPointQueryResult q;
  cudaError_t err = cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q);
  if (err != cudaSuccess || q != cudaDriverEntryPointSuccess || *fn == nullptr)
    return fail(ENGRAM_E_CUDA, "%s entry point unavailable", name);
  return ENGRAM_OK;
}

// Unique id of the current context (0 when none is current).  Ids are never
// reused within a process, unlike CUcontext handle values.
int current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (get_current == nullptr || get_id == nullptr) {
    void* a = nullptr;
    void* b = nullptr;
    int rc = driver_fn("cuCtxGetCurrent", &a);
    if (rc == ENGRAM_OK) rc = driver_fn("cuCtxGetId", &b);
    if (rc) return rc;
    get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    get_id = reinterpret_cast<CtxGetIdFn>(b);
  }
  CUcontext ctx = nullptr;
  *id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS) return fail(ENGRAM_E_CUDA, "cuCtxGetCurrent failed");
  if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return fail(ENGRAM_E_CUDA, "cuCtxGetId failed");
  return ENGRAM_OK;
}

// Device address of g_stage_scratch on the current device.  It is looked up
// (cudaGetSymbolAddress, with the device current) on the first call made on
// a device, and again whenever that device's context has changed since
// (cudaDeviceReset destroys the context and its module; the array may then
// sit elsewhere in the new one).  The check costs two driver queries.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (dev < 0 || dev >= kMaxDevices) return fail(ENGRAM_E_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = 0;
  int rc = current_ctx_id(&id);
  if (rc) return rc;
  if (g_addr[dev] == nullptr || id == 0 || id != g_ctx_id[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_stage_scratch);
    if (err != cudaSuccess || p == nullptr)
      return fail(ENGRAM_E_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(err));
    rc = current_ctx_id(&id);  // the lookup creates the primary context if none was current
    if (rc) return rc;
    g_addr[dev] = p;
    g_ctx_id[dev] = id;
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
