// The original Engram layer's short causal convolution on the gated value,
// fused with the residual add.
//
// Pages cited by title:
//   [P-DETAIL] "DeepSeek Engram 详解：把静态知识从计算里拆出来"
//       §4.2 Short convolution (Y = SiLU(Conv1D(RMSNorm(V~))) + V~, kernel 4,
//       dilation = the largest n-gram order, depthwise and causal),
//       §五 (hidden = hidden + gated + refined) and §9.5 (decode keeps the
//       past (kernel-1)*dilation normalised values).
//   [P-V41] "DeepSeek-V4.1 模型结构（5）：记忆，Engram" §"V4.1 相对原版的两处改动"
//       (the branch V4.1 removed) and §多模态细节 (gate 0 at image positions).
//
// For stream m of position t, with V~ = g * bf16(v):
//   n_t   = gamma^(m) * V~_t / sqrt(mean(V~_t^2) + eps)
//         = gamma^(m) * (r_t * v_t),   r_t = g / sqrt(g^2 * mean(v_t^2) + eps)
//   c_t   = sum_k w[k] * n_{t - k*dilation}          (zeros / carried state before the start)
//   h_t  <- bf16(h_t + (g * v_t + SiLU(c_t)))
//
// Three launches: (1) one warp per position reduces mean(v^2) and writes r
// and the position's sequence; (2) the add streams h once -- a thread owns
// 8 channels of one stream, keeps that stream's filter taps in registers and
// walks a run of consecutive positions, reading the tap positions' v from
// L1/L2 (every v row serves kernel-size positions and hc streams); (3) the
// last (kernel-1)*dilation normalised values of each sequence go to the
// state ring, after (2) has read the old ones.
//
// HBM-bound like the plain gate: per position hc*H bf16 of h read and
// written, H bf16 of v read, the filters once per run of positions.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "engram_internal.h"

namespace engram {
namespace {

constexpr int kMaxK = 4;
constexpr int kMaxHcConv = 8;
constexpr int kMaxRing = 64;
constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ void unpack8(const uint4 x, float (&f)[8]) {
  f[0] = bf16_lo(x.x); f[1] = bf16_hi(x.x);
  f[2] = bf16_lo(x.y); f[3] = bf16_hi(x.y);
  f[4] = bf16_lo(x.z); f[5] = bf16_hi(x.z);
  f[6] = bf16_lo(x.w); f[7] = bf16_hi(x.w);
}

// The normalised value, one expression shared by the add and the state
// writer so that a value read back from the state equals the in-batch one.
__device__ __forceinline__ float normed(float gamma, float r, float v) { return gamma * (r * v); }

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

struct ConvArgs {
  const float* gate;      // [T][hc]
  const uint4* v;         // [T][H/8]
  uint4* h;               // [T][hc][H/8]
  const uint8_t* mask;    // [T] or null
  int64_t n_tokens;
  int hidden, hc;
  const int64_t* cu;      // [n_seqs+1] or null (position t is sequence t)
  int64_t n_seqs;
  const int32_t* slots;   // [n_seqs] or null (identity)
  const float* w;         // [K][hc][H]
  const float* gamma;     // [hc][H]
  int K, dil, ring;       // ring = (K-1)*dil
  float eps;
  float* state;           // [n_slots][ring][hc][H] or null
  int32_t* head;          // [n_slots]
  int64_t n_slots;
  float* r;               // workspace [T][hc]
  int32_t* seq;           // workspace [T]: sequence index, -1 = padding
  int32_t* status;        // or null
};

__device__ __forceinline__ int32_t slot_of(const ConvArgs& a, int64_t s) {
  return a.slots != nullptr ? a.slots[s] : static_cast<int32_t>(s);
}

// (1) r[t][m] and seq[t]; one warp per position.
__global__ void __launch_bounds__(kThreads) conv_prep_kernel(ConvArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  const int nvec = a.hidden / 8;
  for (int64_t t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); t < a.n_tokens; t += warps) {
    float ss = 0.f;
    for (int i = lane; i < nvec; i += 32) {
      float f[8];
      unpack8(__ldg(a.v + t * nvec + i), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const bool masked = a.mask != nullptr && a.mask[t] != 0;
    const float ms = ss / static_cast<float>(a.hidden);
    if (lane < a.hc) {
      const float g = masked ? 0.f : a.gate[t * a.hc + lane];
      a.r[t * a.hc + lane] = g / sqrtf(g * g * ms + a.eps);
    }
    if (lane == 0) {
      int64_t s = t;
      if (a.cu != nullptr) {  // last s with cu[s] <= t
        int64_t lo = 0, hi = a.n_seqs - 1;
        while (lo < hi) {
          const int64_t mid = (lo + hi + 1) >> 1;
          if (a.cu[mid] <= t) lo = mid; else hi = mid - 1;
        }
        s = lo;
      }
      const int32_t slot = slot_of(a, s);
      int32_t out = static_cast<int32_t>(s);
      if (slot < 0) {
        out = -1;  // padding entry
      } else if (a.state != nullptr && slot >= a.n_slots) {
        if (a.status != nullptr) atomicOr(a.status, ENGRAM_ST_BAD_SLOT);
        out = -1;
      }
      a.seq[t] = out;
    }
  }
}

// (2) h <- bf16(h + g v + SiLU(sum_k w[k] n_{t-k*dil})).
__global__ void __launch_bounds__(kThreads) conv_add_kernel(ConvArgs a, int tokens_per_block) {
  const int nchunk = a.hidden / 8;
  const int p = blockIdx.x * kThreads + threadIdx.x;
  if (p >= a.hc * nchunk) return;
  const int m = p / nchunk, c = p - m * nchunk;
  const int i0 = c * 8;
  float w[kMaxK][8], gam[8];
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) {
    if (k < a.K) {
      const float4* wp = reinterpret_cast<const float4*>(a.w + (static_cast<int64_t>(k) * a.hc + m) * a.hidden + i0);
      const float4 x = __ldg(wp), y = __ldg(wp + 1);
      w[k][0] = x.x; w[k][1] = x.y; w[k][2] = x.z; w[k][3] = x.w;
      w[k][4] = y.x; w[k][5] = y.y; w[k][6] = y.z; w[k][7] = y.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) w[k][j] = 0.f;
    }
  }
  {
    const float4* gp = reinterpret_cast<const float4*>(a.gamma + static_cast<int64_t>(m) * a.hidden + i0);
    const float4 x = __ldg(gp), y = __ldg(gp + 1);
    gam[0] = x.x; gam[1] = x.y; gam[2] = x.z; gam[3] = x.w;
    gam[4] = y.x; gam[5] = y.y; gam[6] = y.z; gam[7] = y.w;
  }
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * tokens_per_block;
  const int64_t t1 = t0 + tokens_per_block < a.n_tokens ? t0 + tokens_per_block : a.n_tokens;
  for (int64_t t = t0; t < t1; ++t) {
    const int32_t s = a.seq[t];
    if (s < 0) continue;
    const int64_t start = a.cu != nullptr ? a.cu[s] : t;
    const int64_t local = t - start;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    float vt[8];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      if (k >= a.K) break;
      const int64_t ql = local - static_cast<int64_t>(k) * a.dil;
      float n[8];
      if (ql >= 0) {
        const int64_t q = start + ql;
        const float rq = a.r[q * a.hc + m];
        float f[8];
        unpack8(__ldg(a.v + q * nchunk + c), f);
        if (k == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j) vt[j] = f[j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) n[j] = normed(gam[j], rq, f[j]);
      } else if (a.state != nullptr) {
        const int32_t slot = slot_of(a, s);
        int64_t idx = (static_cast<int64_t>(a.head[slot]) + ql) % a.ring;
        if (idx < 0) idx += a.ring;
        const float4* sp = reinterpret_cast<const float4*>(
            a.state + ((static_cast<int64_t>(slot) * a.ring + idx) * a.hc + m) * a.hidden + i0);
        const float4 x = sp[0], y = sp[1];
        n[0] = x.x; n[1] = x.y; n[2] = x.z; n[3] = x.w;
        n[4] = y.x; n[5] = y.y; n[6] = y.z; n[7] = y.w;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) n[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(w[k][j], n[j], acc[j]);
    }
    const bool masked = a.mask != nullptr && a.mask[t] != 0;
    const float g = masked ? 0.f : a.gate[t * a.hc + m];
    uint4* hp = a.h + (t * a.hc + m) * nchunk + c;
    const uint4 hv = *hp;
    float hf[8];
    unpack8(hv, hf);
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = hf[j] + (g * vt[j] + silu(acc[j]));
    uint4 out;
    out.x = pack_bf16(o[0], o[1]);
    out.y = pack_bf16(o[2], o[3]);
    out.z = pack_bf16(o[4], o[5]);
    out.w = pack_bf16(o[6], o[7]);
    *hp = out;
  }
}

// (3) state ring: the last min(ring, len) normalised values of each sequence,
// then head <- (head + len) mod ring.  One block per sequence.
__global__ void __launch_bounds__(kThreads) conv_state_kernel(ConvArgs a) {
  const int64_t s = blockIdx.x;
  const int32_t slot = slot_of(a, s);
  if (slot < 0 || slot >= a.n_slots) return;
  const int64_t start = a.cu != nullptr ? a.cu[s] : s;
  const int64_t len = a.cu != nullptr ? a.cu[s + 1] - start : 1;
  const int64_t first = len > a.ring ? len - a.ring : 0;
  const int32_t head = a.head[slot];
  const int nchunk = a.hidden / 8;
  const int64_t per_pos = static_cast<int64_t>(a.hc) * nchunk;
  const int64_t work = (len - first) * per_pos;
  for (int64_t x = threadIdx.x; x < work; x += blockDim.x) {
    const int64_t local = first + x / per_pos;
    const int rem = static_cast<int>(x - (local - first) * per_pos);
    const int m = rem / nchunk, c = rem - m * nchunk;
    const int64_t t = start + local;
    const float rq = a.r[t * a.hc + m];
    float f[8];
    unpack8(__ldg(a.v + t * nchunk + c), f);
    const float* gp = a.gamma + static_cast<int64_t>(m) * a.hidden + c * 8;
    float n[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) n[j] = normed(__ldg(gp + j), rq, f[j]);
    const int64_t idx = (static_cast<int64_t>(head) + local) % a.ring;
    float4* sp = reinterpret_cast<float4*>(a.state + ((static_cast<int64_t>(slot) * a.ring + idx) * a.hc + m) *
                                                         a.hidden + c * 8);
    sp[0] = make_float4(n[0], n[1], n[2], n[3]);
    sp[1] = make_float4(n[4], n[5], n[6], n[7]);
  }
  if (threadIdx.x == 0) a.head[slot] = static_cast<int32_t>((head + len) % a.ring);
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" size_t engram_short_conv_workspace_bytes(int64_t n_tokens, int32_t hc) {
  if (n_tokens < 0 || hc < 1) return 0;
  return round256(static_cast<size_t>(n_tokens) * hc * sizeof(float)) +
         round256(static_cast<size_t>(n_tokens) * sizeof(int32_t));
}

extern "C" int engram_short_conv_add(const float* gate_d, const uint16_t* v_d, uint16_t* h_d,
                                     const uint8_t* mask_d, int64_t n_tokens, int32_t hidden, int32_t hc,
                                     const int64_t* cu_seqlens_d, int64_t n_seqs, const int32_t* slots_d,
                                     const float* conv_w_d, const float* gamma_d, int32_t kernel_size,
                                     int32_t dilation, float eps, float* state_d, int32_t* state_head_d,
                                     int64_t n_slots, void* workspace_d, size_t workspace_bytes,
                                     int32_t* status_d, void* stream) {
  if (n_tokens < 0 || n_seqs < 0) return fail(ENGRAM_E_INVALID, "negative size");
  if (hidden < 256 || hidden % 256 != 0) return fail(ENGRAM_E_SHAPE, "hidden %d % 256 != 0", hidden);
  if (hc < 1 || hc > kMaxHcConv) return fail(ENGRAM_E_SHAPE, "hc %d not in [1, %d]", hc, kMaxHcConv);
  if (kernel_size < 1 || kernel_size > kMaxK) return fail(ENGRAM_E_SHAPE, "kernel_size %d not in [1, %d]",
                                                          kernel_size, kMaxK);
  if (dilation < 1) return fail(ENGRAM_E_SHAPE, "dilation %d < 1", dilation);
  const int ring = (kernel_size - 1) * dilation;
  if (ring > kMaxRing) return fail(ENGRAM_E_SHAPE, "(kernel_size-1)*dilation = %d > %d", ring, kMaxRing);
  if (!(eps >= 0.f)) return fail(ENGRAM_E_INVALID, "eps must be >= 0");
  if (cu_seqlens_d == nullptr && n_seqs != n_tokens)
    return fail(ENGRAM_E_SHAPE, "without cu_seqlens every position is its own sequence (n_seqs == n_tokens)");
  if (cu_seqlens_d != nullptr && n_seqs < 1 && n_tokens > 0) return fail(ENGRAM_E_SHAPE, "n_seqs < 1");
  if (state_d != nullptr && (state_head_d == nullptr || n_slots < 1))
    return fail(ENGRAM_E_INVALID, "a state needs its head array and n_slots >= 1");
  if (state_d != nullptr && ring == 0) state_d = nullptr;  // kernel 1 keeps no past
  if (n_tokens == 0) return ENGRAM_OK;
  if (!gate_d || !v_d || !h_d || !conv_w_d || !gamma_d || !workspace_d)
    return fail(ENGRAM_E_INVALID, "null device pointer");
  if (!aligned(v_d, 16) || !aligned(h_d, 16) || !aligned(conv_w_d, 16) || !aligned(gamma_d, 16) ||
      !aligned(workspace_d, 256) || (state_d && !aligned(state_d, 16)))
    return fail(ENGRAM_E_ALIGN, "v, h, conv_w, gamma, state 16-byte and workspace 256-byte aligned");
  if (workspace_bytes < engram_short_conv_workspace_bytes(n_tokens, hc))
    return fail(ENGRAM_E_RANGE, "workspace too small");
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;

  ConvArgs a;
  a.gate = gate_d;
  a.v = reinterpret_cast<const uint4*>(v_d);
  a.h = reinterpret_cast<uint4*>(h_d);
  a.mask = mask_d;
  a.n_tokens = n_tokens;
  a.hidden = hidden;
  a.hc = hc;
  a.cu = cu_seqlens_d;
  a.n_seqs = n_seqs;
  a.slots = slots_d;
  a.w = conv_w_d;
  a.gamma = gamma_d;
  a.K = kernel_size;
  a.dil = dilation;
  a.ring = ring > 0 ? ring : 1;
  a.eps = eps;
  a.state = state_d;
  a.head = state_head_d;
  a.n_slots = state_d ? n_slots : 0;
  a.r = static_cast<float*>(workspace_d);
  a.seq = reinterpret_cast<int32_t*>(static_cast<char*>(workspace_d) +
                                     round256(static_cast<size_t>(n_tokens) * hc * sizeof(float)));
  a.status = status_d;
  cudaStream_t st = as_stream(stream);

  const int64_t warps_needed = n_tokens;
  const int64_t prep_cap = static_cast<int64_t>(sms) * 8;
  const int64_t prep_blocks = (warps_needed + 7) / 8 < prep_cap ? (warps_needed + 7) / 8 : prep_cap;
  conv_prep_kernel<<<static_cast<int>(prep_blocks), kThreads, 0, st>>>(a);
  rc = check_launch("conv_prep_kernel");
  if (rc) return rc;

  const int pairs = hc * (hidden / 8);
  const int gx = (pairs + kThreads - 1) / kThreads;
  int tpb = 32;  // positions per block: fewer when that leaves SMs idle
  while (tpb > 1 && static_cast<int64_t>(gx) * ((n_tokens + tpb - 1) / tpb) < 4LL * sms) tpb >>= 1;
  const int64_t gy = (n_tokens + tpb - 1) / tpb;
  if (gy > 65535) {
    tpb = static_cast<int>((n_tokens + 65534) / 65535);
  }
  const dim3 grid(gx, static_cast<unsigned>((n_tokens + tpb - 1) / tpb));
  conv_add_kernel<<<grid, kThreads, 0, st>>>(a, tpb);
  rc = check_launch("conv_add_kernel");
  if (rc) return rc;

  if (state_d != nullptr) {
    if (n_seqs > 0x7fffffff) return fail(ENGRAM_E_RANGE, "too many sequences");
    conv_state_kernel<<<static_cast<unsigned>(n_seqs), kThreads, 0, st>>>(a);
    rc = check_launch("conv_state_kernel");
  }
  return rc;
}
