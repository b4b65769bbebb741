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
//   n_t   = gamma^(m) * V~_t / sqrt(mean(V~_t^2) + eps) = gamma^(m) * x_t,
//   x_t   = r_t * v_t,   r_t = g / sqrt(g^2 * mean(v_t^2) + eps)
//   c_t   = sum_k (w[k] * gamma^(m)) * x_{t - k*dilation}   (zeros / carried state before the start)
//   h_t  <- bf16(h_t + (g * v_t + SiLU(c_t)))
//
// Three launches: (1) one warp per position reduces mean(v^2) and writes r,
// the position's sequence and its index in it; (2) the add streams h once
// (see conv_add_kernel); (3) the last (kernel-1)*dilation values x of each
// sequence go to the state ring, after (2) has read the old ones.
//
// HBM-bound like the plain gate: per position hc*H bf16 of h read and
// written, H bf16 of v read, the filters once per run of positions.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

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


__device__ __forceinline__ uint64_t f2_bf16(uint32_t w) {  // the two bf16 of a word, widened
  return f2(bf16_lo(w), bf16_hi(w));
}

// x * sigmoid(x) = x / (1 + 2^(-x log2 e)) of both lanes of a packed pair,
// with the hardware base-2 exponential and reciprocal approximations (PTX
// ex2.approx.ftz.f32, rcp.approx.ftz.f32; each about 2^-22 relative): a few
// ulp plus about 1.2 |x| ulp from rounding the exponent's argument.  Inputs
// below -126/log2 e give 2^(..) = inf and a result of -0, the limit of
// x sigmoid(x).
__device__ __forceinline__ uint64_t silu2(uint64_t x) {
  float m0, m1, e0, e1, d0, d1, r0, r1;
  f2_split(f2_mul(x, f2(-1.4426950408889634f, -1.4426950408889634f)), m0, m1);
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(m0));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(m1));
  f2_split(f2_add(f2(1.0f, 1.0f), f2(e0, e1)), d0, d1);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d0));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d1));
  return f2_mul(x, f2(r0, r1));
}

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
  float* ge;              // workspace [T][hc]: the gate, 0 at masked positions
  int32_t* seq;           // workspace [T]: sequence index, -1 = padding
  int32_t* pos;           // workspace [T]: index within the sequence, -1 = padding
  int32_t* head0;         // workspace [T]: at a sequence's first position, its slot's ring head on entry
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
      a.ge[t * a.hc + lane] = g;
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
      const int64_t local = t - (a.cu != nullptr ? a.cu[s] : t);
      a.pos[t] = out < 0 ? -1 : static_cast<int32_t>(local);
      // the ring head as it was on entry, for the state writer (which
      // advances it while other blocks still need the old value)
      if (out >= 0 && local == 0 && a.state != nullptr) a.head0[t] = a.head[slot];
    }
  }
}

// (2) h <- bf16(h + g v + SiLU(sum_k (w[k] gamma) x_{t-k*dil})), x_q = r_q v_q.
//
// A thread owns 8 channels of one stream (the filter taps, with gamma folded
// in, stay in registers); a warp owns 256 consecutive channels of one stream,
// so for every position its h and v are one contiguous 512-byte segment each.
// A block walks one residue class mod dilation of a run of positions:
// t, t+dil, t+2*dil, ...  Along the walk the taps of position t are the x of
// the walk's previous positions, so x is computed once per position and kept
// in a register window of three slots used round-robin (the loop is unrolled
// three times, so the slots are fixed registers).  Positions at least
// (K-1)*dil into their sequence take a branch-free path; the others read the
// taps that fall before the sequence start from the state ring (or zero).
//
// Loads are per warp and asynchronous: lane 0 keeps the h and v segments of
// the next kInStages-1 positions of the walk in flight as bulk copies into
// the warp's shared-memory ring (one mbarrier per stage); results go out as
// one coalesced 512-byte store per warp.
constexpr int kInStages = 8;
constexpr int kCh = 8;                    // channels per thread
constexpr int kWarps = kThreads / 32;
constexpr int kSegBytes = 32 * kCh * 2;   // 512
struct WarpRing {
  uint4 h[kInStages][32];
  uint4 v[kInStages][32];
  uint64_t bar[kInStages];
};

// A bounded wait that polls without the suspend hint of mbar_wait_bounded.
// Each warp of the convolution waits once per position for copies issued
// seven positions earlier, which have almost always landed; polling is 1.5 %
// faster there (0.555 vs 0.564 ms for the 16,384-token stage).
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > kWaitBudgetCycles) return false;
  }
}

template <int K>
__global__ void __launch_bounds__(kThreads, 2) conv_add_kernel(ConvArgs a, int walk_len) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WarpRing& wr = reinterpret_cast<WarpRing*>(smem_raw)[warp];
  const int nchunk = a.hidden / kCh;
  const int p = blockIdx.x * kThreads + threadIdx.x;
  // hidden % 256 == 0, so a warp never straddles two streams and either all
  // of its lanes have work or none has
  if (p - lane >= a.hc * nchunk) return;
  const int m = p / nchunk, c = p - m * nchunk;
  const int hc = a.hc, dil = a.dil;
  constexpr int kP = kCh / 2;  // channel pairs per thread
  uint64_t wg[K][kP];           // filter taps with the RMSNorm weight folded in, packed pairs
  {
    const float4* gq = reinterpret_cast<const float4*>(a.gamma + static_cast<int64_t>(m) * a.hidden + c * kCh);
    const float4 gx = __ldg(gq), gy = __ldg(gq + 1);
    const float gam[8] = {gx.x, gx.y, gx.z, gx.w, gy.x, gy.y, gy.z, gy.w};
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const float4* wp = reinterpret_cast<const float4*>(a.w + (static_cast<int64_t>(k) * hc + m) * a.hidden + c * kCh);
      const float4 x = __ldg(wp), y = __ldg(wp + 1);
      const float wk[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
      for (int j = 0; j < kP; ++j) wg[k][j] = f2(wk[2 * j] * gam[2 * j], wk[2 * j + 1] * gam[2 * j + 1]);
    }
  }
  // this block's walk: positions t0 + rho + j*dil, j < walk_len, below t1
  const int rho = static_cast<int>(blockIdx.y % static_cast<unsigned>(dil));
  const int64_t span = static_cast<int64_t>(walk_len) * dil;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y / static_cast<unsigned>(dil)) * span;
  const int64_t t1 = t0 + span < a.n_tokens ? t0 + span : a.n_tokens;
  const int64_t first = t0 + rho;
  const int n_pos = first < t1 ? static_cast<int>((t1 - first + dil - 1) / dil) : 0;
  if (n_pos == 0) return;

  // strides in 16-byte units along the walk
  const int64_t hstride = static_cast<int64_t>(hc) * nchunk * dil;
  const int64_t vstride = static_cast<int64_t>(nchunk) * dil;
  const uint4* hsrc = a.h + (first * hc + m) * nchunk + (c - lane);  // the warp's segment at `first`
  const uint4* vsrc = a.v + first * nchunk + (c - lane);
  uint4* hdst = a.h + (first * hc + m) * nchunk + c;
  const float* rp = a.r + first * hc + m;  // advanced along the walk
  const float* gp = a.ge + first * hc + m;
  const int32_t* pp = a.pos + first;
  const int64_t sstride = static_cast<int64_t>(hc) * dil;  // r and ge along the walk

  if (lane == 0) {
    for (int s = 0; s < kInStages; ++s) mbar_init(smem_u32(&wr.bar[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  int ji = 0;           // next walk index to fetch
  uint32_t issued = 0;  // stages with a copy in flight (lane 0)
  auto issue = [&](int s) {
    if (ji < n_pos) {
      if (lane == 0) {
        const uint32_t bar = smem_u32(&wr.bar[s]);
        mbar_arrive_expect_tx(bar, 2 * kSegBytes);
        bulk_g2s(smem_u32(&wr.h[s][0]), hsrc + ji * hstride, kSegBytes, bar);
        bulk_g2s(smem_u32(&wr.v[s][0]), vsrc + ji * vstride, kSegBytes, bar);
        issued |= 1u << s;
      }
      ++ji;
    }
  };
  for (int s = 0; s < kInStages - 1; ++s) issue(s);

  // window slot (u - k) mod 3 holds x of k steps back at unrolled step u (packed pairs)
  uint64_t win[3][kP];
#pragma unroll
  for (int k = 1; k <= 3; ++k) {
    const int64_t q = first - static_cast<int64_t>(k) * dil;
    uint64_t* wdst = win[(3 - k) % 3];
    if (k < K && q >= 0) {
      const float rq = __ldg(a.r + q * hc + m);
      const uint4 vq = __ldg(a.v + q * nchunk + c);
      const uint32_t vw[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
      for (int j = 0; j < kP; ++j) wdst[j] = f2_mul(f2(rq, rq), f2_bf16(vw[j]));
    } else {
#pragma unroll
      for (int j = 0; j < kP; ++j) wdst[j] = f2(0.f, 0.f);
    }
  }

  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  float rt = __ldg(rp), gt = __ldg(gp);
  int32_t lt = __ldg(pp);
  const int64_t tail = static_cast<int64_t>(K - 1) * dil;  // positions before this take the general path
  int j = 0;
  while (true) {
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      if (j >= n_pos) goto done;
      issue(stage == 0 ? kInStages - 1 : stage - 1);
      {
        const bool landed = mbar_wait_spin(smem_u32(&wr.bar[stage]), (phase >> stage) & 1u);
        if (!__all_sync(0xffffffffu, landed)) {  // uniform, so no lane is left at a barrier
          ok = false;
          goto done;
        }
      }
      phase ^= 1u << stage;
      if (lane == 0) issued &= ~(1u << stage);
      {
        const uint4 hv = wr.h[stage][lane], vv = wr.v[stage][lane];
        __syncwarp();  // every lane has read in-stage `stage` before lane 0 refills it
        // next position's scalars
        float rt_n = 0.f, gt_n = 0.f;
        int32_t lt_n = -1;
        rp += sstride;
        gp += sstride;
        pp += dil;
        if (j + 1 < n_pos) {
          rt_n = __ldg(rp);
          gt_n = __ldg(gp);
          lt_n = __ldg(pp);
        }
        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
        uint64_t xt[kP];
        {
          const uint64_t rt2 = f2(rt, rt);
#pragma unroll
          for (int q = 0; q < kP; ++q) xt[q] = f2_mul(rt2, f2_bf16(vw[q]));
        }
        if (lt >= 0) {
          uint64_t acc[kP];
#pragma unroll
          for (int q = 0; q < kP; ++q) acc[q] = f2_mul(wg[0][q], xt[q]);
          if (lt >= tail) {
#pragma unroll
            for (int k = 1; k < K; ++k) {
#pragma unroll
              for (int q = 0; q < kP; ++q) acc[q] = f2_fma(wg[k][q], win[(u - k + 3) % 3][q], acc[q]);
            }
          } else {
#pragma unroll
            for (int k = 1; k < K; ++k) {
              const int ql = lt - k * dil;
              if (ql >= 0) {
#pragma unroll
                for (int q = 0; q < kP; ++q) acc[q] = f2_fma(wg[k][q], win[(u - k + 3) % 3][q], acc[q]);
              } else if (a.state != nullptr) {
                const int64_t tc = first + static_cast<int64_t>(j) * dil;
                const int64_t t_start = tc - lt;  // the sequence's first position
                const int32_t slot = slot_of(a, a.seq[tc]);
                int64_t idx = (static_cast<int64_t>(a.head0[t_start]) + ql) % a.ring;
                if (idx < 0) idx += a.ring;
                const float4* sp = reinterpret_cast<const float4*>(
                    a.state + ((static_cast<int64_t>(slot) * a.ring + idx) * hc + m) * a.hidden + c * kCh);
                const float4 x = sp[0], y = sp[1];
                const uint64_t sx[4] = {f2(x.x, x.y), f2(x.z, x.w), f2(y.x, y.y), f2(y.z, y.w)};
#pragma unroll
                for (int q = 0; q < kP; ++q) acc[q] = f2_fma(wg[k][q], sx[q], acc[q]);
              }
            }
          }
          // h + (g v + SiLU(c)), a pair of channels at a time
          const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
          const uint64_t gt2 = f2(gt, gt);
          uint32_t ow[4];
#pragma unroll
          for (int q = 0; q < kP; ++q) {
            float lo, hi;
            f2_split(f2_add(f2_bf16(hw[q]), f2_fma(gt2, f2_bf16(vw[q]), silu2(acc[q]))), lo, hi);
            ow[q] = pack_bf16(lo, hi);
          }
          *hdst = make_uint4(ow[0], ow[1], ow[2], ow[3]);  // padding positions are not written
        }
        hdst += hstride;
        // the window slot of x_t is the one that held x of three steps back
#pragma unroll
        for (int q = 0; q < kP; ++q) win[u][q] = xt[q];
        rt = rt_n;
        gt = gt_n;
        lt = lt_n;
      }
      stage = stage + 1 == kInStages ? 0 : stage + 1;
      ++j;
    }
  }
done:
  if (lane == 0 && !ok) {
    if (a.status != nullptr) atomicOr(a.status, ENGRAM_ST_TIMEOUT);
    // let the copies still in flight land before the shared memory is released
    for (int s = 0; s < kInStages; ++s)
      if (issued & (1u << s)) mbar_wait_bounded(smem_u32(&wr.bar[s]), (phase >> s) & 1u, nullptr);
  }
  __syncwarp();
}

// (3) state ring: the last min(ring, len) values x of each sequence, then
// head <- (head + len) mod ring.  One block per (sequence, kept position);
// the entry head comes from the prep kernel's copy, so the block that
// advances the head races with no reader.
__global__ void __launch_bounds__(kThreads) conv_state_kernel(ConvArgs a) {
  const int64_t s = blockIdx.x;
  const int32_t slot = slot_of(a, s);
  if (slot < 0 || slot >= a.n_slots) return;
  const int64_t start = a.cu != nullptr ? a.cu[s] : s;
  const int64_t len = a.cu != nullptr ? a.cu[s + 1] - start : 1;
  const int64_t keep = len < a.ring ? len : a.ring;
  if (static_cast<int64_t>(blockIdx.y) >= keep) return;
  const int64_t local = len - keep + blockIdx.y;
  const int32_t head = a.head0[start];
  const int nchunk = a.hidden / 8;
  const int per_pos = a.hc * nchunk;
  const int64_t t = start + local;
  const int64_t idx = (static_cast<int64_t>(head) + local) % a.ring;
  for (int x = threadIdx.x; x < per_pos; x += blockDim.x) {
    const int m = x / nchunk, c = x - m * nchunk;
    const float rq = a.r[t * a.hc + m];
    float f[8];
    unpack8(__ldg(a.v + t * nchunk + c), f);
    float n[8];  // the same product as the add's window, so state taps equal in-batch taps
#pragma unroll
    for (int j = 0; j < 8; ++j) n[j] = rq * f[j];
    float4* sp = reinterpret_cast<float4*>(a.state + ((static_cast<int64_t>(slot) * a.ring + idx) * a.hc + m) *
                                                         a.hidden + c * 8);
    sp[0] = make_float4(n[0], n[1], n[2], n[3]);
    sp[1] = make_float4(n[4], n[5], n[6], n[7]);
  }
  if (blockIdx.y == 0 && threadIdx.x == 0) a.head[slot] = static_cast<int32_t>((head + len) % a.ring);
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

template <int K>
int launch_add(dim3 grid, int smem, cudaStream_t st, const ConvArgs& a, int walk) {
  static std::atomic<uint64_t> attr_set{0};  // one bit per device: the shared-memory opt-in was made
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(attr_set.load(std::memory_order_relaxed) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(conv_add_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    attr_set.fetch_or(bit, std::memory_order_relaxed);
  }
  conv_add_kernel<K><<<grid, kThreads, smem, st>>>(a, walk);
  return check_launch("conv_add_kernel");
}

int launch_conv_add(int K, dim3 grid, int smem, cudaStream_t st, const ConvArgs& a, int walk) {
  switch (K) {
    case 1: return launch_add<1>(grid, smem, st, a, walk);
    case 2: return launch_add<2>(grid, smem, st, a, walk);
    case 3: return launch_add<3>(grid, smem, st, a, walk);
    default: return launch_add<4>(grid, smem, st, a, walk);
  }
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" size_t engram_short_conv_workspace_bytes(int64_t n_tokens, int32_t hc) {
  if (n_tokens < 0 || hc < 1) return 0;
  return 2 * round256(static_cast<size_t>(n_tokens) * hc * sizeof(float)) +
         3 * round256(static_cast<size_t>(n_tokens) * sizeof(int32_t));
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
  a.ge = reinterpret_cast<float*>(static_cast<char*>(workspace_d) +
                                  round256(static_cast<size_t>(n_tokens) * hc * sizeof(float)));
  a.seq = reinterpret_cast<int32_t*>(static_cast<char*>(workspace_d) +
                                     2 * round256(static_cast<size_t>(n_tokens) * hc * sizeof(float)));
  a.pos = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(a.seq) +
                                     round256(static_cast<size_t>(n_tokens) * sizeof(int32_t)));
  a.head0 = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(a.pos) +
                                       round256(static_cast<size_t>(n_tokens) * sizeof(int32_t)));
  a.status = status_d;
  cudaStream_t st = as_stream(stream);

  const int64_t warps_needed = n_tokens;
  const int64_t prep_cap = static_cast<int64_t>(sms) * 8;
  const int64_t prep_blocks = (warps_needed + 7) / 8 < prep_cap ? (warps_needed + 7) / 8 : prep_cap;
  conv_prep_kernel<<<static_cast<int>(prep_blocks), kThreads, 0, st>>>(a);
  rc = check_launch("conv_prep_kernel");
  if (rc) return rc;

  const int pairs = hc * (hidden / kCh);
  const int gx = (pairs + kThreads - 1) / kThreads;
  // a block walks walk_len positions of one residue class; shorter walks
  // when the grid would leave SMs idle, longer ones to stay within grid.y
  int walk = 32;
  auto blocks_y = [&](int wl) {
    return ((n_tokens + static_cast<int64_t>(wl) * dilation - 1) / (static_cast<int64_t>(wl) * dilation)) * dilation;
  };
  while (walk > 1 && static_cast<int64_t>(gx) * blocks_y(walk) < 4LL * sms) walk >>= 1;
  while (blocks_y(walk) > 65535) walk <<= 1;
  const dim3 grid(gx, static_cast<unsigned>(blocks_y(walk)));
  const int smem = static_cast<int>(sizeof(WarpRing)) * kWarps;
  rc = launch_conv_add(kernel_size, grid, smem, st, a, walk);
  if (rc) return rc;

  if (state_d != nullptr) {
    if (n_seqs > 0x7fffffff) return fail(ENGRAM_E_RANGE, "too many sequences");
    conv_state_kernel<<<dim3(static_cast<unsigned>(n_seqs), static_cast<unsigned>(ring)), kThreads, 0, st>>>(a);
    rc = check_launch("conv_state_kernel");
  }
  return rc;
}
