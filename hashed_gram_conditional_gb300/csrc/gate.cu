// Stage 5b/5c of the Engram lookup: finish the context gate from the
// projection's partial sums and apply the gated residual add in place.
//
// Pages cited by title:
//   [P-V41] "DeepSeek-V4.1 模型结构（5）：记忆，Engram" §门控 and
//           §"sigmoid 之前多一步带符号的平方根"
//   [P-DS4] "ds4.c 学习笔记" -- glossary entry "Engram", §消费：学习投影 + 余弦门控
//           (h <- bf16(h + gate * bf16(v)); the masked branch returns)
//   [P-O1]  "条件记忆：DeepSeek V4.1 Engram 如何用 O(1) 查表换掉一层计算" §2.3
//           (the gate runs in fp32)
//
// HBM-bound: per position it reads hc*H bf16 of h and H bf16 of v and writes
// hc*H bf16 of h.  A CTA handles 8 positions at a time: each warp reduces one
// position's partial sums in a fixed order (deterministic), then all threads
// stream the 8 rows with 16-byte vectors, reusing each v vector for every
// stream.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "engram_internal.h"

namespace engram {
namespace {

constexpr int kMaxHc = 8;

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t h, float g, uint32_t v) {
  return pack_bf16(bf16_lo(h) + g * bf16_lo(v), bf16_hi(h) + g * bf16_hi(v));
}

// The gate of position t, stream m, from the projection's partial sums
// (reduced over the tiles by the warp's lanes, then across lanes); lane 0
// holds the result.
__device__ __forceinline__ float warp_gate(const float4* __restrict__ partials, int64_t t, int m, int hc, int ntile,
                                           float inv_h, float eps, float clamp, float score_scale) {
  const int lane = threadIdx.x & 31;
  float dot = 0.f, kk = 0.f, hh = 0.f;
  const float4* p = partials + (t * hc + m) * ntile;
  for (int q = lane; q < ntile; q += 32) {
    const float4 x = __ldg(p + q);
    dot += x.x;
    kk += x.y;
    hh += x.z;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    dot += __shfl_xor_sync(0xffffffffu, dot, o);
    kk += __shfl_xor_sync(0xffffffffu, kk, o);
    hh += __shfl_xor_sync(0xffffffffu, hh, o);
  }
  // s = dot * rstd(h) * rstd(k) * scale; gate = sigmoid(signed sqrt(s))
  const float sc = dot * (1.0f / sqrtf(hh * inv_h + eps)) * (1.0f / sqrtf(kk * inv_h + eps)) * score_scale;
  const float z = copysignf(sqrtf(fmaxf(fabsf(sc), clamp)), sc);
  return 1.0f / (1.0f + expf(-z));
}

// A CTA takes P <= 8 positions at a time (P is chosen so that small batches
// still spread over the SMs): warp w < P finishes the gates of position w,
// then all 256 threads stream the P positions' rows (v once, every stream of
// h read and written) with 16-byte vectors.
constexpr int kPosPerCta = 8;

__global__ void __launch_bounds__(256) gate_add_kernel(
    const float4* __restrict__ partials, const uint4* __restrict__ v, uint4* h,
    const uint8_t* __restrict__ mask, int64_t n_tokens, int hidden, int hc, float eps,
    float clamp, float score_scale, float* __restrict__ gate_out, int pos_per_cta) {
  __shared__ float gs[kPosPerCta][kMaxHc];
  __shared__ uint8_t live[kPosPerCta];
  // launched as a programmatic dependent: the partial sums, v and h are read
  // only after the previous kernel (the projection) has finished
  wait_prior_grids();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntile = hidden / 256;
  const int nvec = hidden / 8;  // 16-byte vectors per stream row
  const float inv_h = 1.0f / static_cast<float>(hidden);
  const int P = pos_per_cta;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * P; base < n_tokens;
       base += static_cast<int64_t>(gridDim.x) * P) {
    const int64_t t = base + warp;
    if (warp < P && t < n_tokens) {
      // [P-DS4] step 4: a masked position returns untouched; its gate is 0.
      const bool masked = (mask != nullptr) && mask[t] != 0;
      for (int m = 0; m < hc; ++m) {
        const float g = masked ? 0.f : warp_gate(partials, t, m, hc, ntile, inv_h, eps, clamp, score_scale);
        if (lane == 0) {
          gs[warp][m] = g;
          if (gate_out != nullptr) gate_out[t * hc + m] = g;
        }
      }
      if (lane == 0) live[warp] = masked ? 0 : 1;
    } else if (warp < P && lane == 0) {
      live[warp] = 0;
    }
    __syncthreads();
    if (h != nullptr) {  // no h: gates only
      const int work = P * nvec;
      for (int i = threadIdx.x; i < work; i += blockDim.x) {
        const int p = i / nvec, j = i - p * nvec;
        if (!live[p]) continue;
        const int64_t tp = base + p;
        const uint4 vv = v[tp * nvec + j];
        uint4* ht = h + tp * static_cast<int64_t>(hc) * nvec + j;
        uint4 hv[kMaxHc];
#pragma unroll
        for (int m = 0; m < kMaxHc; ++m)
          if (m < hc) hv[m] = ht[m * nvec];
#pragma unroll
        for (int m = 0; m < kMaxHc; ++m) {
          if (m >= hc) break;
          const float g = gs[p][m];
          uint4 o;
          o.x = fma_bf16x2(hv[m].x, g, vv.x);
          o.y = fma_bf16x2(hv[m].y, g, vv.y);
          o.z = fma_bf16x2(hv[m].z, g, vv.z);
          o.w = fma_bf16x2(hv[m].w, g, vv.w);
          ht[m * nvec] = o;
        }
      }
    }
    __syncthreads();  // gs and live are rewritten for the next 8 positions
  }
}

// The gates alone (no residual): one warp per position.
__global__ void __launch_bounds__(256) gates_kernel(const float4* __restrict__ partials,
                                                    const uint8_t* __restrict__ mask, int64_t n_tokens,
                                                    int hidden, int hc, float eps, float clamp, float score_scale,
                                                    float* __restrict__ gate_out) {
  wait_prior_grids();  // as gate_add_kernel
  const int lane = threadIdx.x & 31;
  const int ntile = hidden / 256;
  const float inv_h = 1.0f / static_cast<float>(hidden);
  const int64_t warps = static_cast<int64_t>(gridDim.x) * 8;
  for (int64_t t = blockIdx.x * 8 + (threadIdx.x >> 5); t < n_tokens; t += warps) {
    const bool masked = (mask != nullptr) && mask[t] != 0;
    for (int m = 0; m < hc; ++m) {
      const float g = masked ? 0.f : warp_gate(partials, t, m, hc, ntile, inv_h, eps, clamp, score_scale);
      if (lane == 0) gate_out[t * hc + m] = g;
    }
  }
}

// 256-thread launch configuration on `st`; set_pdl makes it a programmatic
// dependent of the previous kernel in the stream.
cudaLaunchConfig_t pdl_config(int blocks, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  return cfg;
}
void set_pdl(cudaLaunchAttribute* attr) {
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" int engram_gate_add(const float* partials_d, const uint16_t* v_d, uint16_t* h_d,
                               const uint8_t* mask_d, int64_t n_tokens, int32_t hidden, int32_t hc,
                               float eps, float clamp, float score_scale, float* gate_out_d,
                               void* stream) {
  if (n_tokens < 0) return fail(ENGRAM_E_INVALID, "n_tokens < 0");
  if (hidden < 256 || hidden % 256 != 0) return fail(ENGRAM_E_SHAPE, "hidden %d % 256 != 0", hidden);
  if (hc < 1 || hc > kMaxHc) return fail(ENGRAM_E_SHAPE, "hc %d not in [1, %d]", hc, kMaxHc);
  if (n_tokens == 0) return ENGRAM_OK;
  if (!partials_d) return fail(ENGRAM_E_INVALID, "null partials");
  if (!h_d && !gate_out_d) return fail(ENGRAM_E_INVALID, "gates only (h = NULL) needs gate_out");
  if (h_d && !v_d) return fail(ENGRAM_E_INVALID, "null v");
  if (!aligned(partials_d, 16) || (h_d && (!aligned(v_d, 16) || !aligned(h_d, 16))))
    return fail(ENGRAM_E_ALIGN, "partials, v and h must be 16-byte aligned");
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  if (h_d == nullptr) {  // gates only
    const int64_t cap = static_cast<int64_t>(sms) * 16;
    const int64_t need = (n_tokens + 7) / 8;
    cudaLaunchConfig_t cfg = pdl_config(static_cast<int>(need < cap ? need : cap), as_stream(stream));
    cudaLaunchAttribute attr;
    cfg.attrs = &attr;
    set_pdl(&attr);
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, gates_kernel, reinterpret_cast<const float4*>(partials_d),
                                               mask_d, n_tokens, hidden, hc, eps, clamp, score_scale, gate_out_d);
    if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "gates_kernel launch: %s", cudaGetErrorString(err));
    return check_launch("gates_kernel");
  }
  // positions per CTA: 8 when there are enough positions for 4 CTAs per SM
  int P = kPosPerCta;
  while (P > 1 && (n_tokens + P - 1) / P < 4LL * sms) P >>= 1;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  const int64_t need = (n_tokens + P - 1) / P;
  const int blocks = static_cast<int>(need < cap ? need : cap);
  cudaLaunchConfig_t cfg = pdl_config(blocks, as_stream(stream));
  cudaLaunchAttribute attr;
  cfg.attrs = &attr;
  set_pdl(&attr);
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, gate_add_kernel, reinterpret_cast<const float4*>(partials_d),
                                             reinterpret_cast<const uint4*>(v_d), reinterpret_cast<uint4*>(h_d),
                                             mask_d, n_tokens, hidden, hc, eps, clamp, score_scale, gate_out_d, P);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "gate_add_kernel launch: %s", cudaGetErrorString(err));
  return check_launch("gate_add_kernel");
}
