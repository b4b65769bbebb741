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
// hc*H bf16 of h.  One CTA handles one position at a time; warp 0 reduces the
// partial sums in a fixed order (deterministic), then all threads stream the
// row with 16-byte vectors, reusing each v vector for every stream.
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

__global__ void __launch_bounds__(256) gate_add_kernel(
    const float4* __restrict__ partials, const uint4* __restrict__ v, uint4* h,
    const uint8_t* __restrict__ mask, int64_t n_tokens, int hidden, int hc, float eps,
    float clamp, float score_scale, float* __restrict__ gate_out) {
  __shared__ float gs[kMaxHc];
  const int ntile = hidden / 256;
  const int nvec = hidden / 8;  // 16-byte vectors per stream row
  const float inv_h = 1.0f / static_cast<float>(hidden);
  for (int64_t t = blockIdx.x; t < n_tokens; t += gridDim.x) {
    const bool masked = (mask != nullptr) && mask[t] != 0;
    if (masked) {
      // [P-DS4] step 4: the masked branch returns; the gate is 0.
      if (gate_out != nullptr && threadIdx.x < hc) gate_out[t * hc + threadIdx.x] = 0.0f;
      continue;
    }
    if (threadIdx.x < 32) {
      const uint32_t lane = threadIdx.x;
      for (int m = 0; m < hc; ++m) {
        float dot = 0.f, kk = 0.f, hh = 0.f;
        const float4* p = partials + (t * hc + m) * ntile;
        for (int q = lane; q < ntile; q += 32) {
          const float4 x = p[q];
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
        if (lane == 0) {
          // s = dot * rstd(h) * rstd(k) * scale; gate = sigmoid(signed sqrt(s))
          const float s = dot * (1.0f / sqrtf(hh * inv_h + eps)) * (1.0f / sqrtf(kk * inv_h + eps)) *
                          score_scale;
          const float z = copysignf(sqrtf(fmaxf(fabsf(s), clamp)), s);
          const float g = 1.0f / (1.0f + expf(-z));
          gs[m] = g;
          if (gate_out != nullptr) gate_out[t * hc + m] = g;
        }
      }
    }
    __syncthreads();
    float g[kMaxHc];
#pragma unroll
    for (int m = 0; m < kMaxHc; ++m) g[m] = (m < hc) ? gs[m] : 0.f;
    const uint4* vt = v + t * nvec;
    uint4* ht = h + t * static_cast<int64_t>(hc) * nvec;
    for (int i = threadIdx.x; h != nullptr && i < nvec; i += blockDim.x) {  // no h: gates only
      const uint4 vv = vt[i];
#pragma unroll
      for (int m = 0; m < kMaxHc; ++m) {
        if (m >= hc) break;
        uint4 hv = ht[m * nvec + i];
        hv.x = fma_bf16x2(hv.x, g[m], vv.x);
        hv.y = fma_bf16x2(hv.y, g[m], vv.y);
        hv.z = fma_bf16x2(hv.z, g[m], vv.z);
        hv.w = fma_bf16x2(hv.w, g[m], vv.w);
        ht[m * nvec + i] = hv;
      }
    }
    __syncthreads();  // gs is rewritten for the next position
  }
}

// The gates alone (no residual): one warp per position, lanes over the
// partials' tiles, streams in turn.
__global__ void __launch_bounds__(256) gates_kernel(const float4* __restrict__ partials,
                                                    const uint8_t* __restrict__ mask, int64_t n_tokens,
                                                    int hidden, int hc, float eps, float clamp, float score_scale,
                                                    float* __restrict__ gate_out) {
  const int lane = threadIdx.x & 31;
  const int ntile = hidden / 256;
  const float inv_h = 1.0f / static_cast<float>(hidden);
  const int64_t warps = static_cast<int64_t>(gridDim.x) * 8;
  for (int64_t t = blockIdx.x * 8 + (threadIdx.x >> 5); t < n_tokens; t += warps) {
    const bool masked = (mask != nullptr) && mask[t] != 0;
    for (int m = 0; m < hc; ++m) {
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
      if (lane == 0) {
        const float sc = dot * (1.0f / sqrtf(hh * inv_h + eps)) * (1.0f / sqrtf(kk * inv_h + eps)) * score_scale;
        const float z = copysignf(sqrtf(fmaxf(fabsf(sc), clamp)), sc);
        gate_out[t * hc + m] = masked ? 0.0f : 1.0f / (1.0f + expf(-z));
      }
    }
  }
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
    gates_kernel<<<static_cast<int>(need < cap ? need : cap), 256, 0, as_stream(stream)>>>(
        reinterpret_cast<const float4*>(partials_d), mask_d, n_tokens, hidden, hc, eps, clamp, score_scale,
        gate_out_d);
    return check_launch("gates_kernel");
  }
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  const int blocks = static_cast<int>(n_tokens < cap ? n_tokens : cap);
  gate_add_kernel<<<blocks, 256, 0, as_stream(stream)>>>(
      reinterpret_cast<const float4*>(partials_d), reinterpret_cast<const uint4*>(v_d),
      reinterpret_cast<uint4*>(h_d), mask_d, n_tokens, hidden, hc, eps, clamp, score_scale,
      gate_out_d);
  return check_launch("gate_add_kernel");
}
