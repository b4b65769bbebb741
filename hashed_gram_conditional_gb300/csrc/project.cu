// Stage 5a/5b of the Engram lookup: kv = e @ wkv on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM, operands staged by TMA), with
// the context gate's reductions fused into the epilogue.
//
// Pages cited by title:
//   [P-V41] "DeepSeek-V4.1 模型结构（5）：记忆，Engram" §门控 (one linear map from
//           the 6144-dim lookup vector to 4 keys and 1 value of 5120 each) and
//           §"每条流一个 key 的设计沿用自原版" (one [6144, 25600] matrix wkv)
//   [P-DS4] "ds4.c 学习笔记" -- glossary entry "Engram", §消费：学习投影 + 余弦门控
//           (dot = sum_i h_i (q_w_i k_w_i) k_i and the two mean squares)
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: 128x64 tile of e and 256x64 tile of the packed
//               wkv per k-block into a 4-stage ring (48 KB per stage, 128-byte
//               swizzle), completion on the stage's "full" mbarrier.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//               issues tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) from one
//               thread; tcgen05.commit frees each stage and, per tile, signals
//               the accumulator to the epilogue.
//   warps 2-5   epilogue: tcgen05.ld 32 columns at a time; thread r owns row r
//               (one position) of the tile.  For a key tile it accumulates, over
//               its 256 columns, sum h q_w k_w k, sum k^2 and sum h^2 into one
//               float4 partial per (position, stream, tile); keys never reach
//               memory.  For a value tile it rounds v to bf16 and stores it.
//   Two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
// Fused mode (engram_project_gate): within each group of M-blocks every key
// tile is scheduled before any value tile.  A key tile's epilogue warps
// publish their partials and bump a per-M-block counter; a value tile's
// epilogue waits (bounded) until all key tiles of its M-block are published,
// forms the gates of its rows from the partials and applies
// h <- bf16(h + g * bf16(v)) directly, so v never reaches memory and the
// residual traffic overlaps tensor work.  The launch is cooperative, so every
// CTA is resident and the wait always ends: the key tiles a value tile needs
// come earlier in the static tile order, and the lowest-numbered waiting tile
// only ever waits on CTAs that are not themselves waiting.
// Every wait is bounded; a wait that runs out records ENGRAM_ST_TIMEOUT, the
// roles unwind, in-flight copies and MMAs are drained and TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdlib>

#include "engram_internal.h"

namespace engram {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int kThreads = 192;
constexpr int kGroupM = 16;  // M-blocks per raster group: e group + wkv wave fit one die's L2 half
// CTA pair (cta_group::2): a 256 x 256 tile per pair; each CTA stages its own
// 128 rows of e and its half (128 rows) of the 256 wkv rows per k-block.
constexpr int STAGES2 = 6;
constexpr int B2_BYTES = (BN / 2) * BK * 2;
constexpr int STAGE2_BYTES = A_BYTES + B2_BYTES;
constexpr int kGroupM2 = 16;  // pair M-blocks (4096 rows) per raster group: the e group (50 MB) stays in L2
constexpr int kMaxHc = 8;

struct ProjArgs {
  int64_t M;
  int32_t K;
  int32_t H;
  int32_t hc;
  int32_t mt;           // 128-row blocks
  int32_t mt2;          // 256-row blocks (CTA-pair kernel)
  int32_t nt;
  int32_t num_tiles;    // tiles of the kernel that runs (128x256 or 256x256)
  uint16_t* h;           // read (key tiles); updated in place by value tiles in fused mode
  const float* q_w;
  const float* k_w;
  float4* partials;
  uint16_t* v;           // unfused mode only
  int32_t* status;
  // fused mode only
  const uint8_t* mask;
  float* gate_out;
  int32_t* cnt;          // [mt][hc][4] published key-tile epilogue warps per (M-block, stream, quarter)
  int32_t* ready;        // [mt] finished (stream, quarter) gate groups per M-block
  int32_t* abort_g;      // one word: a CTA gave up (tells the others to stop waiting)
  float* gates;          // [mt*128][hc] finished gates (-1 = masked row)
  float eps;
  float clamp;
  float score_scale;
};

struct __align__(8) SmemCtl {
  uint64_t full[STAGES2];
  uint64_t empty[STAGES2];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
  float qk[4][BN];            // q_w * k_w of the current key tile, one copy per epilogue warp
  uint32_t sv[4][32][20];     // fused mode: a warp's 32 x 32 bf16 v chunk, rows padded to 80 B
  float sg[4][32][kMaxHc];    // fused mode: gates of the warp's 32 rows (-1 = leave the row alone)
};

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// tile: start address, leading byte offset (unused for this layout, 16 B),
// stride byte offset 1024 B between 8-row groups, descriptor version 1,
// swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B bf16,
// both K-major, N = BN, M = BM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                            (static_cast<uint32_t>(BM >> 4) << 24);
// Same for the CTA pair: M = 256 (128 rows per CTA), N = 256.
constexpr uint32_t kIdesc2 = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                             (static_cast<uint32_t>((2 * BM) >> 4) << 24);

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}


// 32 lanes x 16 columns of 32-bit TMEM words, waited for.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- CTA-pair primitives
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 2-D TMA load into this CTA's shared memory whose completion is counted on
// the mbarrier at cluster address `bar` (the leader CTA's barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 4-D tiled TMA loads of the packed wkv ([N/128][K/64][128][64]).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int32_t c2, int32_t c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(tmap), "r"(0), "r"(0), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const void* tmap, int32_t c2, int32_t c3,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5}], [%6];" ::"r"(dst),
      "l"(tmap), "r"(0), "r"(0), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc2), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at this shared offset in both CTAs of the pair
// when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(static_cast<unsigned short>(3))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

__device__ __forceinline__ void tile_coords(int tile, int mt, int nt, int group, int& mb, int& nb) {
  const int per_group = group * nt;
  const int g = tile / per_group;
  const int first_m = g * group;
  const int gm = min(group, mt - first_m);
  const int local = tile - g * per_group;
  mb = first_m + local % gm;
  nb = local / gm;
}

__device__ __forceinline__ void raise_abort(SmemCtl* ctl, const ProjArgs& a) {
  ctl->abort = 1;
  if (a.abort_g) atomicExch(a.abort_g, 1);  // tell the other CTAs (fused mode)
  if (a.status) atomicOr(a.status, static_cast<int>(ENGRAM_ST_TIMEOUT));
}

// Waits until *cnt >= target (acquire), bounded; false on timeout or abort.
__device__ bool wait_published(const int32_t* cnt, int target, const volatile int32_t* global_abort,
                               const volatile int* cta_abort) {
  const long long t0 = clock64();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) return true;
    if (*global_abort || *cta_abort) return false;
    if (clock64() - t0 > kWaitBudgetCycles) return false;
    __nanosleep(64);
  }
}

// Diagnostic: a wait that nothing will satisfy gives up after the budget and
// records ENGRAM_ST_TIMEOUT (engram_selftest_wait).
__global__ void selftest_wait_kernel(int which, int32_t* scratch, int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int cta_abort;
  if (threadIdx.x != 0) return;
  bool ok;
  if (which == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    ok = mbar_wait_bounded(smem_u32(&bar), 0, nullptr);  // phase 0 never completes
  } else {
    cta_abort = 0;
    ok = wait_published(scratch, 1, scratch + 1, &cta_abort);  // the counter stays 0
  }
  if (!ok && status != nullptr) atomicOr(status, static_cast<int>(ENGRAM_ST_TIMEOUT));
}

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Two bf16 lanes of h and v: bf16_rne(h + g * v) in fp32 per lane.
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t h, float g, uint32_t v) {
  const float lo = __uint_as_float(h << 16) + g * __uint_as_float(v << 16);
  const float hi = __uint_as_float(h & 0xffff0000u) + g * __uint_as_float(v & 0xffff0000u);
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Tile geometry shared by the epilogue helpers.
struct EpiTile {
  int m;         // key stream of a key tile
  int c0;        // first column of the tile within its key stream / within v
  bool key_tile;
};

__device__ __forceinline__ EpiTile epi_tile(const ProjArgs& a, int nb) {
  EpiTile e;
  const int n0 = nb * BN;
  const int key_cols = a.hc * a.H;
  e.key_tile = n0 < key_cols;
  e.m = e.key_tile ? n0 / a.H : 0;
  e.c0 = e.key_tile ? n0 - e.m * a.H : n0 - key_cols;
  return e;
}

// Asks L2 for `bytes` (a multiple of 16) at a 16-byte-aligned global address.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Before the accumulator is ready: ask L2 for the h row segments the key
// tile's epilogue will read (each lane its own row: 256 columns of the key's
// stream, 512 B), so that the epilogue's loads hit L2 rather than each chunk
// waiting on DRAM; and stage q_w * k_w of the tile's 256 columns in the
// warp's own copy (no cross-warp barrier).
__device__ __forceinline__ void epilogue_stage(const ProjArgs& a, SmemCtl* ctl, int q, uint32_t lane, int mb,
                                               const EpiTile& et) {
  if (!et.key_tile) return;
  const int64_t t = static_cast<int64_t>(mb) * BM + q * 32 + static_cast<int>(lane);
  if (t < a.M) l2_prefetch(a.h + (t * a.hc + et.m) * a.H + et.c0, BN * 2);
  float* qk = ctl->qk[q];
  __syncwarp();
  for (int c = static_cast<int>(lane); c < BN; c += 32) {
    const int64_t idx = static_cast<int64_t>(et.c0 + c) * a.hc + et.m;
    qk[c] = __ldg(a.q_w + idx) * __ldg(a.k_w + idx);
  }
  __syncwarp();
}

// Epilogue of one 128 x 256 accumulator (TMEM address taddr of this warp's
// 32 lanes): output rows mb*128 + q*32 + lane, columns nb*256 .. +255.
// Returns false when a bounded wait gave up.
template <bool kFuse>
__device__ __forceinline__ bool epilogue_tile(const ProjArgs& a, SmemCtl* ctl, int q, uint32_t lane,
                                              uint32_t taddr, int mb, const EpiTile& et,
                                              const volatile int* abort_flag) {
  const int row = q * 32 + static_cast<int>(lane);
  const int ntile = a.H / BN;
  const bool key_tile = et.key_tile;
  const int m = et.m;
  const int c0 = et.c0;
  const float* qk = ctl->qk[q];
  const int64_t t = static_cast<int64_t>(mb) * BM + row;
  const bool live = t < a.M;
  if (key_tile) {
    const uint4* hrow = reinterpret_cast<const uint4*>(a.h + (t * a.hc + m) * a.H + c0);
    float dot = 0.f, kk = 0.f, hh = 0.f;
    // h of chunks ch+1 and ch+2 is in flight while chunk ch is processed
    uint4 hn1[4], hn2[4];
    if (live) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hn1[i] = __ldg(hrow + i);
        hn2[i] = __ldg(hrow + 4 + i);
      }
    }
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      uint4 hv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hv[i] = hn1[i];
        hn1[i] = hn2[i];
      }
      if (live && ch + 2 < BN / 32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) hn2[i] = __ldg(hrow + (ch + 2) * 4 + i);
      }
      uint32_t r[32];
      __syncwarp();
      tc_ld32(taddr + ch * 32, r);
      if (live) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w4[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int col = ch * 32 + i * 8 + j * 2;
            const float h0 = bf16f(w4[j] & 0xffffu), h1 = bf16f(w4[j] >> 16);
            const float k0 = __uint_as_float(r[i * 8 + j * 2]);
            const float k1 = __uint_as_float(r[i * 8 + j * 2 + 1]);
            dot += h0 * qk[col] * k0 + h1 * qk[col + 1] * k1;
            kk += k0 * k0 + k1 * k1;
            hh += h0 * h0 + h1 * h1;
          }
        }
      }
    }
    if (live) a.partials[(t * a.hc + m) * ntile + c0 / BN] = make_float4(dot, kk, hh, 0.f);
    if (kFuse) {
      // Publish this warp's 32 partials; the warp that publishes the last
      // tile of (M-block, stream, row quarter) finishes those 32 gates.
      __threadfence();
      __syncwarp();
      int prev = 0;
      if (lane == 0) prev = atomicAdd(a.cnt + (static_cast<int64_t>(mb) * a.hc + m) * 4 + q, 1);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == ntile - 1) {
        __threadfence();  // acquire: every tile's partials of these rows are visible
        if (live) {
          const bool masked = a.mask != nullptr && a.mask[t] != 0;
          float g = 0.0f;
          if (!masked) {
            const float4* p = a.partials + (t * a.hc + m) * ntile;
            float sd = 0.f, sk = 0.f, sh = 0.f;
            for (int q0 = 0; q0 < ntile; q0 += 24) {  // 24 loads in flight: one round trip at hidden <= 6144
              float4 x[24];
#pragma unroll
              for (int i = 0; i < 24; ++i)
                x[i] = (q0 + i < ntile) ? __ldcg(p + q0 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int i = 0; i < 24; ++i) {  // tile order: deterministic
                sd += x[i].x;
                sk += x[i].y;
                sh += x[i].z;
              }
            }
            const float inv_h = 1.0f / static_cast<float>(a.H);
            const float sc = sd * (1.0f / sqrtf(sh * inv_h + a.eps)) * (1.0f / sqrtf(sk * inv_h + a.eps)) *
                             a.score_scale;
            const float z = copysignf(sqrtf(fmaxf(fabsf(sc), a.clamp)), sc);
            g = 1.0f / (1.0f + expf(-z));
          }
          a.gates[t * a.hc + m] = masked ? -1.0f : g;
          if (a.gate_out != nullptr) a.gate_out[t * a.hc + m] = g;
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(a.ready + mb, 1);
      }
    }
  } else if (kFuse) {
    // ---- value tile, fused: wait for the M-block's gates, then h <- bf16(h + g bf16(v)).
    // The transposed pass gives lane l the 16-byte segment (l & 3) of rows
    // rl = 8 k8 + l / 4; h of those rows is written only by this tile, so the
    // first chunk's h is requested before the gates are, and every later
    // chunk's h one chunk ahead of its update (streams 0..3; more streams use
    // a plain loop).
    const int seg = static_cast<int>(lane & 3);
    const int hc4 = a.hc < 4 ? a.hc : 4;
    uint4 hn[4][4];
    auto load_chunk = [&](int ch, uint4 (&dst)[4][4]) {
#pragma unroll
      for (int k8 = 0; k8 < 4; ++k8) {
        const int64_t tr = static_cast<int64_t>(mb) * BM + q * 32 + k8 * 8 + static_cast<int>(lane >> 2);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < hc4 && tr < a.M)
            dst[k8][j] = *reinterpret_cast<const uint4*>(a.h + (tr * a.hc + j) * a.H + c0 + ch * 32 + seg * 8);
      }
    };
    load_chunk(0, hn);
    bool ready = true;
    if (lane == 0) ready = wait_published(a.ready + mb, 4 * a.hc, a.abort_g, abort_flag);
    ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
    if (!ready) {
      if (lane == 0 && !*abort_flag) raise_abort(ctl, a);
      return false;
    }
    for (int mm = 0; mm < a.hc; ++mm) ctl->sg[q][lane][mm] = live ? __ldcg(a.gates + t * a.hc + mm) : -1.0f;
    __syncwarp();
    uint32_t(*sv)[20] = ctl->sv[q];
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      uint4 hv[4][4];
#pragma unroll
      for (int k8 = 0; k8 < 4; ++k8)
#pragma unroll
        for (int j = 0; j < 4; ++j) hv[k8][j] = hn[k8][j];
      if (ch + 1 < BN / 32) load_chunk(ch + 1, hn);
      uint32_t r[32];
      __syncwarp();
      tc_ld32(taddr + ch * 32, r);
      // v of this row's 32 columns, rounded to bf16, into the warp's staging rows
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(r[i * 8 + j * 2]),
                                                   __uint_as_float(r[i * 8 + j * 2 + 1]));
          pk[j] = *reinterpret_cast<uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(&sv[lane][i * 4]) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      __syncwarp();
#pragma unroll
      for (int k8 = 0; k8 < 4; ++k8) {
        const int rl = k8 * 8 + static_cast<int>(lane >> 2);
        const int64_t tr = static_cast<int64_t>(mb) * BM + q * 32 + rl;
        const uint4 vv = *reinterpret_cast<const uint4*>(&sv[rl][seg * 4]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float g = ctl->sg[q][rl][j];
          if (j >= hc4 || tr >= a.M || g < 0.0f) continue;
          uint4 x = hv[k8][j];
          x.x = fma_bf16x2(x.x, g, vv.x);
          x.y = fma_bf16x2(x.y, g, vv.y);
          x.z = fma_bf16x2(x.z, g, vv.z);
          x.w = fma_bf16x2(x.w, g, vv.w);
          *reinterpret_cast<uint4*>(a.h + (tr * a.hc + j) * a.H + c0 + ch * 32 + seg * 8) = x;
        }
        // streams beyond the fourth (hidden-connection counts above 4)
        for (int mm = 4; mm < a.hc; ++mm) {
          const float g = ctl->sg[q][rl][mm];
          if (tr >= a.M || g < 0.0f) continue;
          uint4* hp = reinterpret_cast<uint4*>(a.h + (tr * a.hc + mm) * a.H + c0 + ch * 32 + seg * 8);
          uint4 x = *hp;
          x.x = fma_bf16x2(x.x, g, vv.x);
          x.y = fma_bf16x2(x.y, g, vv.y);
          x.z = fma_bf16x2(x.z, g, vv.z);
          x.w = fma_bf16x2(x.w, g, vv.w);
          *hp = x;
        }
      }
    }
  } else {
    uint4* vrow = reinterpret_cast<uint4*>(a.v + t * a.H + c0);
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      uint32_t r[32];
      __syncwarp();
      tc_ld32(taddr + ch * 32, r);
      if (live) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t pk[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(r[i * 8 + j * 2]),
                                                     __uint_as_float(r[i * 8 + j * 2 + 1]));
            pk[j] = *reinterpret_cast<uint32_t*>(&b);
          }
          vrow[ch * 4 + i] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
  }
  return true;
}

template <bool kFuse>
__global__ void __launch_bounds__(kThreads, 1)
    project_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES * A_BYTES;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const int nkb = a.K / BK;
  volatile int* abort_flag = &ctl->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->tfull[i]), 1);
      mbar_init(smem_u32(&ctl->tempty[i]), 4);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // Launched as a programmatic dependent (unfused form): the set-up above
  // overlaps the previous kernel's tail; e, the mask and h are read only
  // after it has finished.
  if (!kFuse) wait_prior_grids();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < a.num_tiles; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, a.mt, a.nt, kGroupM, mb, nb);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1, abort_flag)) {
            if (!*abort_flag) raise_abort(ctl, a);
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          tma_load_2d(smem_u32(smA + s * A_BYTES), &tmA, kb * BK, mb * BM, fb);
          tma_load_4d(smem_u32(smB + s * B_BYTES), &tmB, kb, nb * (BN / 128), fb);
        }
      }
      // Drain: the last STAGES loads issued must have landed before the CTA
      // exits (already true after a normal run, where the MMA consumed them).
      for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
        mbar_wait_bounded(smem_u32(&ctl->full[j % STAGES]), (j / STAGES) & 1, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < a.num_tiles; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t aph = (local >> 1) & 1;
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1, abort_flag)) {
          if (!*abort_flag) raise_abort(ctl, a);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag)) {
            if (!*abort_flag) raise_abort(ctl, a);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smA + s * A_BYTES);
          const uint32_t b0 = smem_u32(smB + s * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            tc_mma(d, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&ctl->empty[s]));
        }
        if (ok) tc_commit(smem_u32(&ctl->tfull[acc]));
      }
      // every MMA issued so far completes before TMEM is released
      tc_commit(smem_u32(&ctl->drain));
      mbar_wait_bounded(smem_u32(&ctl->drain), 0, nullptr);
    }
  } else {
    // ---------------- epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int local = 0;
    for (int tile = blockIdx.x; tile < a.num_tiles; tile += gridDim.x, ++local) {
      int mb, nb;
      tile_coords(tile, a.mt, a.nt, kGroupM, mb, nb);
      const int acc = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      const EpiTile et = epi_tile(a, nb);
      epilogue_stage(a, ctl, q, lane, mb, et);
      if (!mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort_flag)) {
        if (lane == 0 && !*abort_flag) raise_abort(ctl, a);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if (!epilogue_tile<kFuse>(a, ctl, q, lane, taddr, mb, et, abort_flag)) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}


// CTA-pair variant: clusters of 2 CTAs; the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256) reading e rows from both CTAs
// and each CTA's half of the 256 wkv rows, so each SM streams half the wkv
// bytes of the single-CTA kernel through shared memory and can keep 6 stages.
// Both CTAs' loads complete on the even CTA's "full" barrier; MMA completion
// is multicast to both CTAs' "empty" / "tfull" barriers; both CTAs' epilogue
// warps release an accumulator on the even CTA's "tempty" barrier (count 8).
template <bool kFuse>
__global__ void __launch_bounds__(kThreads, 1)
    project2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES2 * A_BYTES;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + STAGES2 * STAGE2_BYTES);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int nkb = a.K / BK;
  volatile int* abort_flag = &ctl->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->tfull[i]), 1);
      mbar_init(smem_u32(&ctl->tempty[i]), 8);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  // Both CTAs' barriers are initialised and their TMEM allocated before any
  // cross-CTA signal.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // Launched as a programmatic dependent (unfused form): the set-up above
  // overlaps the previous kernel's tail; e, the mask and h are read only
  // after it has finished.
  if (!kFuse) wait_prior_grids();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int it = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < a.num_tiles; tile += npairs) {
        int mb2, nb;
        tile_coords(tile, a.mt2, a.nt, kGroupM2, mb2, nb);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES2;
          const uint32_t ph = (it / STAGES2) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1, abort_flag)) {
            if (!*abort_flag) raise_abort(ctl, a);
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * STAGE2_BYTES);
          const uint32_t leader_fb = map_to_cta(fb, 0);
          tma_load_2d_pair(smem_u32(smA + s * A_BYTES), &tmA, kb * BK, mb2 * (2 * BM) + static_cast<int>(rank) * BM,
                           leader_fb);
          tma_load_4d_pair(smem_u32(smB + s * B2_BYTES), &tmB, kb, nb * (BN / 128) + static_cast<int>(rank),
                           leader_fb);
        }
      }
      if (rank == 0) {
        // the last stages issued (both CTAs' halves) have landed before exit
        for (int j = (it > STAGES2 ? it - STAGES2 : 0); j < it; ++j)
          mbar_wait_bounded(smem_u32(&ctl->full[j % STAGES2]), (j / STAGES2) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA only)
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < a.num_tiles; tile += npairs, ++local) {
        const int acc = local & 1;
        const uint32_t aph = (local >> 1) & 1;
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1, abort_flag)) {
          if (!*abort_flag) raise_abort(ctl, a);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES2;
          const uint32_t ph = (it / STAGES2) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag)) {
            if (!*abort_flag) raise_abort(ctl, a);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smA + s * A_BYTES);
          const uint32_t b0 = smem_u32(smB + s * B2_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            tc_mma_pair(d, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit_pair(smem_u32(&ctl->empty[s]));
        }
        if (ok) tc_commit_pair(smem_u32(&ctl->tfull[acc]));
      }
      // every MMA issued so far completes before TMEM is released
      tc_commit_pair(smem_u32(&ctl->drain));
      mbar_wait_bounded(smem_u32(&ctl->drain), 0, nullptr);
    }
  } else {
    // ---------------- epilogue (warps 2..5 of both CTAs; each its own 128 rows)
    const int q = warp & 3;
    const uint32_t leader_tempty0 = map_to_cta(smem_u32(&ctl->tempty[0]), 0);
    const uint32_t leader_tempty1 = map_to_cta(smem_u32(&ctl->tempty[1]), 0);
    int local = 0;
    for (int tile = pair; tile < a.num_tiles; tile += npairs, ++local) {
      int mb2, nb;
      tile_coords(tile, a.mt2, a.nt, kGroupM2, mb2, nb);
      const int mb = mb2 * 2 + static_cast<int>(rank);
      const int acc = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      const EpiTile et = epi_tile(a, nb);
      epilogue_stage(a, ctl, q, lane, mb, et);
      if (!mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort_flag)) {
        if (lane == 0 && !*abort_flag) raise_abort(ctl, a);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if (!epilogue_tile<kFuse>(a, ctl, q, lane, taddr, mb, et, abort_flag)) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? leader_tempty1 : leader_tempty0);
    }
  }

  // No CTA leaves while its partner may still signal its barriers or read its
  // shared memory; then both free their TMEM.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// Block-scaled FP8 projection ([P-O1] §2.3: the released model's projection
// weights are block-FP8 and the table payload is E4M3 with E8M0 scales per
// 32 elements).  The gathered rows enter the tensor cores as they are stored
// (tcgen05.mma kind::mxf8f6f4, E4M3 x E4M3 with an E8M0 scale per 32 elements
// of k on both operands, fp32 accumulation), so there is no bf16 e at all.
//
// One CTA per 128 x 256 tile (one M = 128, N = 256 MMA per K = 32 step),
// k-blocks of 128 bytes (four steps), 4 stages of 48 KB.  The scale factors
// travel with the operands: each stage also holds the k-block's scale words
// of the tile's 128 rows of A and 256 rows of B (TMA, 1.5 KB), and the MMA
// thread copies them into TMEM with tcgen05.cp ahead of the k-block's MMAs
// (the tensor pipe runs a thread's copies and MMAs in issue order).  The
// layout the MMA reads -- lane L, column c, byte k holds the scale of row
// (L mod 32) + 32 c for k-step k (c < 4 for the 128 rows of A, c < 8 for the
// 256 rows of B), the same in every lane quarter (established on GB300 by a
// standalone probe) -- is what tcgen05.cp.32x128b.warpx4 makes of a 512-byte
// image whose 16-byte row r holds the words of rows r, r + 32, r + 64 and
// r + 96; the scale arrays are stored in that order (sf_word_index).  Each
// stage has its own TMEM scale slot, rewritten only after the stage's MMAs
// have completed.  TMEM: the 256-column accumulator plus the slots, which
// leaves no room for a second accumulator: the epilogue stalls the tensor
// pipe from the last MMA of a tile to the accumulator's release, so the
// unfused form keeps that window short (epilogue8_split).  The fused form
// reuses the bf16 kernels' epilogue.
constexpr int BK8 = 128;  // bytes = elements per k-block
constexpr int STAGES8 = 4;
constexpr int A8_BYTES = BM * BK8;
constexpr int B8_BYTES = BN * BK8;
constexpr int SF_A_BYTES = BM * 4;  // a k-block's scale words of 128 rows of A
constexpr int SF_BYTES = SF_A_BYTES + BN * 4;  // ... and of 256 rows of B
constexpr int STAGE8_BYTES = A8_BYTES + B8_BYTES;
constexpr int kThreads8 = 192;  // producer, MMA, 4 epilogue warps
constexpr int kSfCols = 12;     // per scale slot: A (4 columns), B (8 columns)
constexpr int kSfBase = BN;     // scale slots after the accumulator, one per stage
constexpr int TMEM8_COLS = 512;

// kind::mxf8f6f4 instruction descriptor: A and B E4M3, K-major, N = 256,
// M = 128, E8M0 scales, both scale-factor ids = the k-step (byte of the
// scale column); the accumulator is fp32.
__device__ __forceinline__ uint32_t idesc8(uint32_t sf_id) {
  return (sf_id << 4) | ((static_cast<uint32_t>(BN) >> 3) << 17) | (1u << 23) |
         ((static_cast<uint32_t>(BM) >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void tc_mma8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.block32 [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte scale image for tcgen05.cp:
// no swizzle, 8-row core matrices of 128 bytes stored one after another
// (stride byte offset 128 B; the leading byte offset is unused with a single
// core matrix along the row), descriptor version 1.
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  return d;
}

// 32 rows x 128 bits from shared memory into 4 TMEM columns, the same rows in
// each of the four lane quarters (warpx4).  The pair form copies in both CTAs
// of the pair, each from its own shared memory into its own TMEM.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Unfused FP8 projection (partial sums of the key tiles, bf16 v): 10 warps.
// Warp 0 loads operands and scales, warp 1 copies the scales to TMEM and
// issues the MMAs, warps 2..9 are the epilogue, two per lane quarter (warp
// w, numbered e = w + 8 inside the epilogue: quarter e & 3 = w & 3, since a
// warp may only reach TMEM lane quarter w & 3; tile columns half * 128 ..
// +127 with half = (e >> 2) & 1, so each quarter has one warp per half).
// Ten warps leave each thread up to 200 registers, so the epilogue keeps a
// key tile's h in registers without spilling.  The fused form has the
// 6-warp layout of kThreads8.
constexpr int kThreads8u = 320;

// The two halves of a key tile's partial sums meet in shared memory: the
// second half writes its (dot, kk, hh) and arrives on its quarter's barrier
// (32 arrivals per key tile), the first half waits, adds and stores.  Slots
// alternate by key tile.
struct __align__(16) Comb8 {
  float4 v[4][2][32];
  uint64_t bar[4];
};

// The 8-warp epilogue of the unfused FP8 kernels.  The accumulator is
// single-buffered (TMEM also holds the scale slots), so the time from the
// accumulator being ready to its release stalls the tensor pipe.  To keep it
// short, a key tile's h columns are loaded into registers before the
// accumulator is ready; once it is, the warp only reads TMEM and does the
// arithmetic of the partial sums, then releases the accumulator; the two
// halves are combined after that.  Returns early (after raising the abort)
// when a bounded wait gives up.
template <bool kPair>
__device__ __forceinline__ void epilogue8_split(const ProjArgs& a, SmemCtl* ctl, Comb8* comb, int warp,
                                                uint32_t lane, uint32_t tmem_base, int first, int step,
                                                uint32_t rank, uint32_t tempty_bar,
                                                const volatile int* abort_flag) {
  const int q = warp & 3;
  const int half = (warp >> 2) & 1;
  const int cb = half * 128;
  float* qk = ctl->qk[q] + cb;
  const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(cb);
  const int ntile = a.H / BN;
  int local = 0, keys = 0;
  for (int tile = first; tile < a.num_tiles; tile += step, ++local) {
    int mbx, nb;
    if (kPair)
      tile_coords(tile, a.mt2, a.nt, kGroupM2, mbx, nb);
    else
      tile_coords(tile, a.mt, a.nt, kGroupM, mbx, nb);
    const int mb = kPair ? mbx * 2 + static_cast<int>(rank) : mbx;
    const EpiTile et = epi_tile(a, nb);
    const int64_t t = static_cast<int64_t>(mb) * BM + q * 32 + static_cast<int>(lane);
    const bool live = t < a.M;
    uint4 hv[16];
    if (et.key_tile) {
      __syncwarp();
      for (int c = static_cast<int>(lane); c < 128; c += 32) {
        const int64_t idx = static_cast<int64_t>(et.c0 + cb + c) * a.hc + et.m;
        qk[c] = __ldg(a.q_w + idx) * __ldg(a.k_w + idx);
      }
      __syncwarp();
      const uint4* hrow = reinterpret_cast<const uint4*>(a.h + (t * a.hc + et.m) * a.H + et.c0 + cb);
#pragma unroll
      for (int i = 0; i < 16; ++i) hv[i] = live ? __ldg(hrow + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    bool ok = true;
    if (lane == 0) ok = mbar_wait_bounded(smem_u32(&ctl->tfull[0]), local & 1, abort_flag);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) {
      if (lane == 0 && !*abort_flag) raise_abort(ctl, a);
      return;
    }
    tc_fence_after();
    float dot = 0.f, kk = 0.f, hh = 0.f;
    if (et.key_tile) {
      // even and odd columns in the two lanes of packed fp32 sums; TMEM is
      // read 16 columns at a time, which keeps the 64 registers of h plus the
      // working set within the 128 a thread has (spilled values would come
      // back through L1, which the operand loads of the next tile keep busy)
      uint64_t d2 = f2(0.f, 0.f), k2s = f2(0.f, 0.f), h2s = f2(0.f, 0.f);
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16) {
        uint32_t r[16];
        __syncwarp();
        tc_ld16(taddr + c16 * 16, r);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint4 hq = hv[c16 * 2 + i];
          const uint32_t w4[4] = {hq.x, hq.y, hq.z, hq.w};
          const float4 qa = *reinterpret_cast<const float4*>(qk + c16 * 16 + i * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qk + c16 * 16 + i * 8 + 4);
          const uint64_t q2[4] = {f2(qa.x, qa.y), f2(qa.z, qa.w), f2(qb.x, qb.y), f2(qb.z, qb.w)};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t h2 = f2(bf16f(w4[j] & 0xffffu), bf16f(w4[j] >> 16));
            const uint64_t k2 = f2(__uint_as_float(r[i * 8 + j * 2]), __uint_as_float(r[i * 8 + j * 2 + 1]));
            d2 = f2_fma(f2_mul(h2, q2[j]), k2, d2);
            k2s = f2_fma(k2, k2, k2s);
            h2s = f2_fma(h2, h2, h2s);
          }
        }
      }
      float lo, hi;
      f2_split(d2, lo, hi);
      dot = lo + hi;
      f2_split(k2s, lo, hi);
      kk = lo + hi;
      f2_split(h2s, lo, hi);
      hh = lo + hi;
    } else {
      // v rounded to bf16, 16 columns at a time, turned through the warp's
      // 1-KB staging area (32 rows x 32 B, 16-byte halves swapped on every
      // other group of 4 rows against bank conflicts) so that two lanes write
      // each row's 32 contiguous bytes
      uint4* stage = reinterpret_cast<uint4*>(&ctl->sv[0][0][0]) + (warp - 8) * 64;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[32];
        __syncwarp();
        tc_ld32(taddr + ch * 32, r);
#pragma unroll
        for (int hx = 0; hx < 2; ++hx) {
#pragma unroll
          for (int sg = 0; sg < 2; ++sg) {
            uint32_t pk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(r[hx * 16 + sg * 8 + j * 2]),
                                                       __uint_as_float(r[hx * 16 + sg * 8 + j * 2 + 1]));
              pk[j] = *reinterpret_cast<uint32_t*>(&b);
            }
            stage[lane * 2 + (sg ^ ((lane >> 2) & 1))] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int rl = k * 16 + static_cast<int>(lane >> 1);
            const int sg = static_cast<int>(lane & 1);
            const uint4 x = stage[rl * 2 + (sg ^ ((rl >> 2) & 1))];
            const int64_t tr = static_cast<int64_t>(mb) * BM + q * 32 + rl;
            if (tr < a.M)
              *reinterpret_cast<uint4*>(a.v + tr * a.H + et.c0 + cb + ch * 32 + hx * 16 + sg * 8) = x;
          }
          __syncwarp();
        }
      }
    }
    float4* slot = &comb->v[q][keys & 1][lane];
    if (et.key_tile && half == 1) {
      *slot = make_float4(dot, kk, hh, 0.f);
      mbar_arrive(smem_u32(&comb->bar[q]));
    }
    if (et.key_tile && half == 0) {
      // the other half's sums; it releases the accumulator without waiting
      if (lane == 0) ok = mbar_wait_bounded(smem_u32(&comb->bar[q]), keys & 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        if (lane == 0 && !*abort_flag) raise_abort(ctl, a);
        return;
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (kPair)
        mbar_arrive_cluster(tempty_bar);
      else
        mbar_arrive(tempty_bar);
    }
    if (et.key_tile) {
      if (half == 0 && live) {
        const float4 o = *slot;
        a.partials[(t * a.hc + et.m) * ntile + et.c0 / BN] = make_float4(dot + o.x, kk + o.y, hh + o.z, 0.f);
      }
      ++keys;
    }
  }
}

// tmSA: the A scale words [K/128][T128] (four E8M0 bytes: the k-block's four
// 32-element scales of a row, rows in sf_word_index order within each 128);
// tmSB: [K/128][N] words likewise for the rows of wkv^T.
template <bool kFuse>
__global__ void __launch_bounds__(kFuse ? kThreads8 : kThreads8u, 1)
    project8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB, ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES8 * A8_BYTES;
  uint8_t* smS = smem + STAGES8 * STAGE8_BYTES;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smS + STAGES8 * SF_BYTES);
  Comb8* comb = reinterpret_cast<Comb8*>((reinterpret_cast<uintptr_t>(ctl + 1) + 15) & ~uintptr_t(15));
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const int nkb = a.K / BK8;
  volatile int* abort_flag = &ctl->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES8; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->tfull[0]), 1);
    mbar_init(smem_u32(&ctl->tempty[0]), kFuse ? 4 : 8);
    if (!kFuse)
      for (int qq = 0; qq < 4; ++qq) mbar_init(smem_u32(&comb->bar[qq]), 32);
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSA);
    prefetch_tmap(&tmSB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(TMEM8_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (operands)
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < a.num_tiles; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, a.mt, a.nt, kGroupM, mb, nb);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES8;
          const uint32_t ph = (it / STAGES8) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1, abort_flag)) {
            if (!*abort_flag) raise_abort(ctl, a);
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(fb, STAGE8_BYTES + SF_BYTES);
          tma_load_2d(smem_u32(smA + s * A8_BYTES), &tmA, kb * BK8, mb * BM, fb);
          tma_load_4d(smem_u32(smB + s * B8_BYTES), &tmB, kb, nb * (BN / 128), fb);
          tma_load_2d(smem_u32(smS + s * SF_BYTES), &tmSA, mb * BM, kb, fb);
          tma_load_2d(smem_u32(smS + s * SF_BYTES + SF_A_BYTES), &tmSB, nb * BN, kb, fb);
        }
      }
      for (int j = (it > STAGES8 ? it - STAGES8 : 0); j < it; ++j)
        mbar_wait_bounded(smem_u32(&ctl->full[j % STAGES8]), (j / STAGES8) & 1, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < a.num_tiles; tile += gridDim.x, ++local) {
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[0]), (local & 1) ^ 1, abort_flag)) {
          if (!*abort_flag) raise_abort(ctl, a);
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES8;
          const uint32_t ph = (it / STAGES8) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag)) {
            if (!*abort_flag) raise_abort(ctl, a);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smA + s * A8_BYTES);
          const uint32_t b0 = smem_u32(smB + s * B8_BYTES);
          const uint32_t s0 = smem_u32(smS + s * SF_BYTES);
          // the stage's scale slot: A (4 columns), B rows 0..127 and 128..255 (4 each)
          const uint32_t sf = tmem_base + static_cast<uint32_t>(kSfBase + s * kSfCols);
          tc_cp_sf(sf, sf_desc(s0));
          tc_cp_sf(sf + 4u, sf_desc(s0 + SF_A_BYTES));
          tc_cp_sf(sf + 8u, sf_desc(s0 + SF_A_BYTES + 512));
#pragma unroll
          for (int k = 0; k < BK8 / 32; ++k)
            tc_mma8(tmem_base, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc8(static_cast<uint32_t>(k)), sf,
                    sf + 4u, (kb | k) != 0 ? 1u : 0u);
          tc_commit(smem_u32(&ctl->empty[s]));
        }
        if (ok) tc_commit(smem_u32(&ctl->tfull[0]));
      }
      tc_commit(smem_u32(&ctl->drain));
      mbar_wait_bounded(smem_u32(&ctl->drain), 0, nullptr);
    }
  } else if (!kFuse || warp < 6) {
    if constexpr (!kFuse) {
      epilogue8_split<false>(a, ctl, comb, warp + 8, lane, tmem_base, static_cast<int>(blockIdx.x),
                             static_cast<int>(gridDim.x), 0, smem_u32(&ctl->tempty[0]), abort_flag);
    } else {
      // ---------------- epilogue (warps 2..5)
      const int q = warp & 3;
      int local = 0;
      for (int tile = blockIdx.x; tile < a.num_tiles; tile += gridDim.x, ++local) {
        int mb, nb;
        tile_coords(tile, a.mt, a.nt, kGroupM, mb, nb);
        const EpiTile et = epi_tile(a, nb);
        epilogue_stage(a, ctl, q, lane, mb, et);
        if (!mbar_wait_bounded(smem_u32(&ctl->tfull[0]), local & 1, abort_flag)) {
          if (lane == 0 && !*abort_flag) raise_abort(ctl, a);
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        if (!epilogue_tile<kFuse>(a, ctl, q, lane, taddr, mb, et, abort_flag)) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[0]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM8_COLS)
                 : "memory");
  }
}

// CTA-pair form of the FP8 projection: clusters of 2 CTAs, the even CTA
// issuing tcgen05.mma.cta_group::2.kind::mxf8f6f4 (M = 256, N = 256).  Each
// CTA streams its 128 e rows and its half of the pair's 256 wkv rows per
// k-block (6 stages of 32 KB, completion on the even CTA's barrier), so each
// SM moves half the wkv bytes of project8_kernel through shared memory.  Each
// CTA's TMEM holds the scales of its own 128 rows of A (4 columns) and of all
// 256 rows of B (8 columns), in the layout of project8_kernel (established by
// a standalone probe on GB300): each CTA loads those scale words into its
// stage, and the even CTA's tcgen05.cp.cta_group::2 copies each CTA's image
// into its own TMEM.  Accumulator single-buffered.
constexpr int STAGES82 = 6;
constexpr int B82_BYTES = (BN / 2) * BK8;
constexpr int STAGE82_BYTES = A8_BYTES + B82_BYTES;


__device__ __forceinline__ void tc_mma8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.block32 [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// M = 256 for the pair.
__device__ __forceinline__ uint32_t idesc82(uint32_t sf_id) {
  return (sf_id << 4) | ((static_cast<uint32_t>(BN) >> 3) << 17) | (1u << 23) |
         ((static_cast<uint32_t>(2 * BM) >> 4) << 24) | (sf_id << 29);
}

template <bool kFuse>
__global__ void __launch_bounds__(kFuse ? kThreads8 : kThreads8u, 1)
    project82_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB, ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES82 * A8_BYTES;
  uint8_t* smS = smem + STAGES82 * STAGE82_BYTES;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smS + STAGES82 * SF_BYTES);
  Comb8* comb = reinterpret_cast<Comb8*>((reinterpret_cast<uintptr_t>(ctl + 1) + 15) & ~uintptr_t(15));
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int nkb = a.K / BK8;
  volatile int* abort_flag = &ctl->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES82; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->tfull[0]), 1);
    mbar_init(smem_u32(&ctl->tempty[0]), kFuse ? 8 : 16);
    if (!kFuse)
      for (int qq = 0; qq < 4; ++qq) mbar_init(smem_u32(&comb->bar[qq]), 32);
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSA);
    prefetch_tmap(&tmSB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(TMEM8_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int it = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < a.num_tiles; tile += npairs) {
        int mb2, nb;
        tile_coords(tile, a.mt2, a.nt, kGroupM2, mb2, nb);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES82;
          const uint32_t ph = (it / STAGES82) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1, abort_flag)) {
            if (!*abort_flag) raise_abort(ctl, a);
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (STAGE82_BYTES + SF_BYTES));
          const uint32_t leader_fb = map_to_cta(fb, 0);
          const int m0 = mb2 * (2 * BM) + static_cast<int>(rank) * BM;
          tma_load_2d_pair(smem_u32(smA + s * A8_BYTES), &tmA, kb * BK8, m0, leader_fb);
          tma_load_4d_pair(smem_u32(smB + s * B82_BYTES), &tmB, kb, nb * (BN / 128) + static_cast<int>(rank),
                           leader_fb);
          // this CTA's 128 rows of A scales, all 256 rows of B scales
          tma_load_2d_pair(smem_u32(smS + s * SF_BYTES), &tmSA, m0, kb, leader_fb);
          tma_load_2d_pair(smem_u32(smS + s * SF_BYTES + SF_A_BYTES), &tmSB, nb * BN, kb, leader_fb);
        }
      }
      if (rank == 0) {
        for (int j = (it > STAGES82 ? it - STAGES82 : 0); j < it; ++j)
          mbar_wait_bounded(smem_u32(&ctl->full[j % STAGES82]), (j / STAGES82) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA only)
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < a.num_tiles; tile += npairs, ++local) {
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[0]), (local & 1) ^ 1, abort_flag)) {
          if (!*abort_flag) raise_abort(ctl, a);
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES82;
          const uint32_t ph = (it / STAGES82) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag)) {
            if (!*abort_flag) raise_abort(ctl, a);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smA + s * A8_BYTES);
          const uint32_t b0 = smem_u32(smB + s * B82_BYTES);
          const uint32_t s0 = smem_u32(smS + s * SF_BYTES);
          const uint32_t sf = tmem_base + static_cast<uint32_t>(kSfBase + s * kSfCols);
          tc_cp_sf_pair(sf, sf_desc(s0));
          tc_cp_sf_pair(sf + 4u, sf_desc(s0 + SF_A_BYTES));
          tc_cp_sf_pair(sf + 8u, sf_desc(s0 + SF_A_BYTES + 512));
#pragma unroll
          for (int k = 0; k < BK8 / 32; ++k)
            tc_mma8_pair(tmem_base, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc82(static_cast<uint32_t>(k)),
                         sf, sf + 4u, (kb | k) != 0 ? 1u : 0u);
          tc_commit_pair(smem_u32(&ctl->empty[s]));
        }
        if (ok) tc_commit_pair(smem_u32(&ctl->tfull[0]));
      }
      tc_commit_pair(smem_u32(&ctl->drain));
      mbar_wait_bounded(smem_u32(&ctl->drain), 0, nullptr);
    }
  } else if (!kFuse || warp < 6) {
    if constexpr (!kFuse) {
      epilogue8_split<true>(a, ctl, comb, warp + 8, lane, tmem_base, pair, npairs, rank,
                            map_to_cta(smem_u32(&ctl->tempty[0]), 0), abort_flag);
    } else {
      // ---------------- epilogue (warps 2..5 of both CTAs; each its own 128 rows)
      const int q = warp & 3;
      const uint32_t leader_tempty = map_to_cta(smem_u32(&ctl->tempty[0]), 0);
      int local = 0;
      for (int tile = pair; tile < a.num_tiles; tile += npairs, ++local) {
        int mb2, nb;
        tile_coords(tile, a.mt2, a.nt, kGroupM2, mb2, nb);
        const int mb = mb2 * 2 + static_cast<int>(rank);
        const EpiTile et = epi_tile(a, nb);
        epilogue_stage(a, ctl, q, lane, mb, et);
        if (!mbar_wait_bounded(smem_u32(&ctl->tfull[0]), local & 1, abort_flag)) {
          if (lane == 0 && !*abort_flag) raise_abort(ctl, a);
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        if (!epilogue_tile<kFuse>(a, ctl, q, lane, taddr, mb, et, abort_flag)) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(leader_tempty);
      }
    }
  }

  // No CTA leaves while its partner may still signal its barriers or read its
  // shared memory; then both free their TMEM.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM8_COLS)
                 : "memory");
  }
}

// Block-FP8 wkv into the operand layouts of project8_kernel: codes [K][N]
// (kv = e @ wkv) -> [N/128][K/128][128][128] bytes, so each 128 x 128-byte
// tile of wkv^T is 16 KB contiguous; scales [K/32][N] -> [K/128][N] words,
// byte j of word (kb, n) = scale of rows kb*128 + 32 j .. +31 of column n,
// the words of each 128 columns in tcgen05.cp image order (sf_word_index).
__global__ void pack_wkv8_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ sf, int64_t K,
                                 int64_t N, uint8_t* __restrict__ wt, uint32_t* __restrict__ sft) {
  __shared__ uint8_t tile[32][33];
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 32, k0 = static_cast<int64_t>(blockIdx.y) * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t k = k0 + r, n = n0 + threadIdx.x;
    tile[r][threadIdx.x] = (k < K && n < N) ? w[k * N + n] : 0;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t n = n0 + r, k = k0 + threadIdx.x;
    if (n < N && k < K)
      wt[(((n / 128) * (K / 128) + k / 128) * 128 + n % 128) * 128 + k % 128] = tile[threadIdx.x][r];
  }
  // scale words: the blocks with threadIdx.y == 0 of the first k-row of every 128 k
  if (blockIdx.y % 4 == 0 && threadIdx.y == 0) {
    const int64_t n = n0 + threadIdx.x, kb = k0 / 128;
    if (n < N && kb < K / 128) {
      uint32_t word = 0;
      for (int j = 0; j < 4; ++j) word |= static_cast<uint32_t>(sf[(kb * 4 + j) * N + n]) << (8 * j);
      sft[kb * N + sf_word_index(n)] = word;
    }
  }
}

// wkv [K][N] -> tiled K-major operand layout [N/128][K/64][128][64]: the
// 128 x 64 tile (rows n, columns k) of every k-block is 16 KB contiguous and a
// 128-row block of wkv^T is one contiguous 1.5 MB run, so operand loads stream
// whole DRAM pages instead of 128-byte pieces of rows 12 KB apart.
__global__ void pack_wkv_kernel(const uint16_t* __restrict__ w, int64_t K, int64_t N,
                                uint16_t* __restrict__ wt) {
  __shared__ uint16_t tile[32][33];
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t k = k0 + i, n = n0 + threadIdx.x;
    if (k < K && n < N) tile[i][threadIdx.x] = w[k * N + n];
  }
  __syncthreads();
  const int64_t kblocks = K / 64;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t n = n0 + i, k = k0 + threadIdx.x;
    if (k < K && n < N) {
      const int64_t idx = (((n >> 7) * kblocks + (k >> 6)) << 13) + ((n & 127) << 6) + (k & 63);
      wt[idx] = tile[threadIdx.x][i];
    }
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int get_encode_fn(EncodeTiledFn* out) {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                       cudaEnableDefault, &q);
    if (err != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr)
      return fail(ENGRAM_E_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  *out = fn;
  return ENGRAM_OK;
}

// 2-D bf16 tensor [rows][cols] (cols contiguous), box = box_rows x 64 columns,
// 128-byte swizzle, zero fill outside the tensor.
int make_tmap(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = nullptr;
  int rc = get_encode_fn(&enc);
  if (rc) return rc;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ENGRAM_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return ENGRAM_OK;
}

// Packed wkv as a 4-D tensor {64, 128, K/64, N/128} (innermost first); a box
// covers one k-block of `nblocks` consecutive 128-row blocks, 128-byte swizzle.
int make_tmap_wkv(CUtensorMap* tm, const void* base, uint64_t N, uint64_t K, uint32_t nblocks) {
  EncodeTiledFn enc = nullptr;
  int rc = get_encode_fn(&enc);
  if (rc) return rc;
  const cuuint64_t dims[4] = {64, 128, K / 64, N / 128};
  const cuuint64_t strides[3] = {128, 128 * 128, (K / 64) * 128 * 128};
  const cuuint32_t box[4] = {64, 128, 1, nblocks};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ENGRAM_E_CUDA, "cuTensorMapEncodeTiled(wkv) failed (%d)", static_cast<int>(r));
  return ENGRAM_OK;
}

// 2-D byte tensor [rows][cols] (E4M3 e), box = box_rows x 128 bytes, 128-byte swizzle.
int make_tmap8(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = nullptr;
  int rc = get_encode_fn(&enc);
  if (rc) return rc;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK8), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ENGRAM_E_CUDA, "cuTensorMapEncodeTiled(e8) failed (%d)", static_cast<int>(r));
  return ENGRAM_OK;
}

// Packed FP8 wkv as a 4-D byte tensor {128, 128, K/128, N/128}; a box covers
// one k-block of `nblocks` consecutive 128-row blocks.
int make_tmap_wkv8(CUtensorMap* tm, const void* base, uint64_t N, uint64_t K, uint32_t nblocks) {
  EncodeTiledFn enc = nullptr;
  int rc = get_encode_fn(&enc);
  if (rc) return rc;
  const cuuint64_t dims[4] = {128, 128, K / 128, N / 128};
  const cuuint64_t strides[3] = {128, 128 * 128, (K / 128) * 128 * 128};
  const cuuint32_t box[4] = {128, 128, 1, nblocks};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ENGRAM_E_CUDA, "cuTensorMapEncodeTiled(wkv8) failed (%d)", static_cast<int>(r));
  return ENGRAM_OK;
}

// Scale words as a 2-D uint32 tensor [rows][cols] (cols contiguous); a box is
// box_cols consecutive words of one row, no swizzle.
int make_tmap_sf(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols) {
  EncodeTiledFn enc = nullptr;
  int rc = get_encode_fn(&enc);
  if (rc) return rc;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {box_cols, 1};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ENGRAM_E_CUDA, "cuTensorMapEncodeTiled(scales) failed (%d)", static_cast<int>(r));
  return ENGRAM_OK;
}

size_t project_smem_bytes(bool pair) {
  return 1024 + (pair ? STAGES2 * STAGE2_BYTES : STAGES * STAGE_BYTES) + sizeof(SmemCtl);
}

// The CTA-pair kernel is the default from 129 tokens on.  A batch of at most
// 128 tokens (one 128-row block) runs the single-CTA kernel: the pair's second
// CTA would hold no rows, and as 128 x 256 tiles the column tiles fill the SMs
// in one wave where the pairs need two (GB300, hidden 5120, 128 tokens, after
// writing a buffer larger than L2: 72 us single-CTA vs 87 us pair).
// engram_kernel_options.projection_cta selects either kernel at every size.
bool use_pair_kernel(int64_t n_tokens) {
  const int forced = kernel_options().projection_cta;
  if (forced != 0) return forced == 2;
  return n_tokens > BM;
}

// Shared argument checks and set-up of both projection entry points.
int prepare(const uint16_t* e_d, int64_t n_tokens, int64_t K, const uint16_t* wkv_packed_d, int32_t hidden,
            int32_t hc, const uint16_t* h_d, const float* q_w_d, const float* k_w_d, float* partials_d,
            int32_t* status_d, bool pair, ProjArgs* a, CUtensorMap* tmA, CUtensorMap* tmB) {
  if (n_tokens < 0) return fail(ENGRAM_E_INVALID, "n_tokens < 0");
  if (K < BK || K % BK != 0 || K > (int64_t(1) << 20))
    return fail(ENGRAM_E_SHAPE, "K %lld must be a positive multiple of 64", (long long)K);
  if (hidden < BN || hidden % BN != 0) return fail(ENGRAM_E_SHAPE, "hidden %d must be a multiple of 256", hidden);
  if (hc < 1 || hc > kMaxHc) return fail(ENGRAM_E_SHAPE, "hc %d not in [1, %d]", hc, kMaxHc);
  if (n_tokens == 0) return ENGRAM_OK;
  if (n_tokens > (int64_t(1) << 31) - 2 * BM) return fail(ENGRAM_E_SHAPE, "too many tokens");
  if (!e_d || !wkv_packed_d || !h_d || !q_w_d || !k_w_d || !partials_d)
    return fail(ENGRAM_E_INVALID, "null device pointer");
  if (!aligned(e_d, 16) || !aligned(wkv_packed_d, 16) || !aligned(h_d, 16) || !aligned(partials_d, 16))
    return fail(ENGRAM_E_ALIGN, "e, wkv, h and partials must be 16-byte aligned");
  int rc = check_device(nullptr);
  if (rc) return rc;
  const int64_t N = static_cast<int64_t>(hc + 1) * hidden;
  if ((rc = make_tmap(tmA, e_d, static_cast<uint64_t>(n_tokens), static_cast<uint64_t>(K), BM))) return rc;
  if ((rc = make_tmap_wkv(tmB, wkv_packed_d, static_cast<uint64_t>(N), static_cast<uint64_t>(K), pair ? 1 : 2)))
    return rc;
  *a = ProjArgs{};
  a->M = n_tokens;
  a->K = static_cast<int32_t>(K);
  a->H = hidden;
  a->hc = hc;
  a->mt = static_cast<int32_t>((n_tokens + BM - 1) / BM);
  a->mt2 = static_cast<int32_t>((n_tokens + 2 * BM - 1) / (2 * BM));
  a->nt = static_cast<int32_t>(N / BN);
  const int64_t tiles = static_cast<int64_t>(pair ? a->mt2 : a->mt) * a->nt;
  if (tiles > INT32_MAX) return fail(ENGRAM_E_SHAPE, "too many tiles");
  a->num_tiles = static_cast<int32_t>(tiles);
  a->h = const_cast<uint16_t*>(h_d);
  a->q_w = q_w_d;
  a->k_w = k_w_d;
  a->partials = reinterpret_cast<float4*>(partials_d);
  a->status = status_d;
  return ENGRAM_OK;
}

// Fused launches are cooperative unless engram_kernel_options.plain_launch
// is set (for profilers that cannot replay a cooperative cluster launch).
// The grid never exceeds the resident capacity either way, and every
// in-kernel wait is bounded.
bool use_cooperative() { return kernel_options().plain_launch == 0; }

using KernelFn = void (*)(CUtensorMap, CUtensorMap, ProjArgs);

// Launches one of the four projection kernels: single CTA or CTA pair,
// unfused or fused.  Fused launches are cooperative (every CTA resident).
int launch(bool pair, bool fused, const CUtensorMap& tmA, const CUtensorMap& tmB, const ProjArgs& a,
           cudaStream_t st) {
  const void* fn = pair ? (fused ? reinterpret_cast<const void*>(&project2_kernel<true>)
                                 : reinterpret_cast<const void*>(&project2_kernel<false>))
                        : (fused ? reinterpret_cast<const void*>(&project_kernel<true>)
                                 : reinterpret_cast<const void*>(&project_kernel<false>));
  const size_t smem = project_smem_bytes(pair);
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaFuncSetAttribute(project): %s", cudaGetErrorString(err));
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  int units = sms;  // CTAs (single) or CTA pairs that can be resident at once
  if (pair) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = 2;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
    cfg.gridDim = dim3(2 * (sms / 2));
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    int clusters = 0;
    err = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg);
    if (err != cudaSuccess || clusters < 1)
      return fail(ENGRAM_E_CUDA, "no resident CTA pair for the projection: %s", cudaGetErrorString(err));
    units = clusters;
  }
  if (fused && use_cooperative()) {
    attr[nattr].id = cudaLaunchAttributeCooperative;
    attr[nattr].val.cooperative = 1;
    ++nattr;
  }
  if (!fused) {  // the unfused kernels wait for the previous grid in-kernel
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  const int n = a.num_tiles < units ? a.num_tiles : units;
  cfg.gridDim = dim3(pair ? 2 * n : n);
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  err = cudaLaunchKernelEx(&cfg, reinterpret_cast<KernelFn>(const_cast<void*>(fn)), tmA, tmB, a);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "project kernel launch: %s", cudaGetErrorString(err));
  return check_launch("project kernel");
}

// The single-CTA FP8 kernel is the default.  The CTA pair moves a third fewer
// operand bytes per SM, but the per-SM MMA rate is the same (an M = 256 pair
// MMA takes as many cycles as an M = 128 one), both issue the same three
// scale copies per k-block per SM, and both keep a single accumulator: on
// 16,384 tokens the two measure within 2 % of each other (1.80-1.82 ms), and
// at 128 tokens the single CTA's 100 tiles fit one wave (43 vs 59 us for
// projection + gate).  engram_kernel_options.fp8_pair selects the pair.
bool use_fp8_pair() { return kernel_options().fp8_pair != 0; }

// Argument checks and set-up of the FP8 entry points.
// tm[0..3]: e8, packed wkv8, A scales, B scales.
int prepare8(const uint8_t* e8_d, const uint32_t* sfa_d, int64_t n_tokens, int64_t K, const uint8_t* w8_d,
             const uint32_t* sfb_d, int32_t hidden, int32_t hc, const uint16_t* h_d, const float* q_w_d,
             const float* k_w_d, float* partials_d, int32_t* status_d, bool pair, ProjArgs* a, CUtensorMap* tm) {
  if (n_tokens < 0) return fail(ENGRAM_E_INVALID, "n_tokens < 0");
  if (K < BK8 || K % BK8 != 0 || K > (int64_t(1) << 20))
    return fail(ENGRAM_E_SHAPE, "K %lld must be a positive multiple of 128", (long long)K);
  if (hidden < BN || hidden % BN != 0) return fail(ENGRAM_E_SHAPE, "hidden %d must be a multiple of 256", hidden);
  if (hc < 1 || hc > kMaxHc) return fail(ENGRAM_E_SHAPE, "hc %d not in [1, %d]", hc, kMaxHc);
  if (n_tokens == 0) return ENGRAM_OK;
  if (n_tokens > (int64_t(1) << 31) - 2 * BM) return fail(ENGRAM_E_SHAPE, "too many tokens");
  if (!e8_d || !sfa_d || !w8_d || !sfb_d || !h_d || !q_w_d || !k_w_d || !partials_d)
    return fail(ENGRAM_E_INVALID, "null device pointer");
  if (!aligned(e8_d, 16) || !aligned(w8_d, 16) || !aligned(h_d, 16) || !aligned(partials_d, 16) ||
      !aligned(sfa_d, 16) || !aligned(sfb_d, 16))
    return fail(ENGRAM_E_ALIGN, "e8, wkv8, h, partials and the scales must be 16-byte aligned");
  int rc = check_device(nullptr);
  if (rc) return rc;
  const int64_t N = static_cast<int64_t>(hc + 1) * hidden;
  const uint64_t t128 = static_cast<uint64_t>((n_tokens + 127) / 128 * 128);
  if ((rc = make_tmap8(&tm[0], e8_d, static_cast<uint64_t>(n_tokens), static_cast<uint64_t>(K), BM))) return rc;
  if ((rc = make_tmap_wkv8(&tm[1], w8_d, static_cast<uint64_t>(N), static_cast<uint64_t>(K), pair ? 1 : 2)))
    return rc;
  if ((rc = make_tmap_sf(&tm[2], sfa_d, static_cast<uint64_t>(K / BK8), t128, BM))) return rc;
  if ((rc = make_tmap_sf(&tm[3], sfb_d, static_cast<uint64_t>(K / BK8), static_cast<uint64_t>(N), BN))) return rc;
  *a = ProjArgs{};
  a->M = n_tokens;
  a->K = static_cast<int32_t>(K);
  a->H = hidden;
  a->hc = hc;
  a->mt = static_cast<int32_t>((n_tokens + BM - 1) / BM);
  a->mt2 = static_cast<int32_t>((n_tokens + 2 * BM - 1) / (2 * BM));
  a->nt = static_cast<int32_t>(N / BN);
  const int64_t tiles = static_cast<int64_t>(pair ? a->mt2 : a->mt) * a->nt;
  if (tiles > INT32_MAX) return fail(ENGRAM_E_SHAPE, "too many tiles");
  a->num_tiles = static_cast<int32_t>(tiles);
  a->h = const_cast<uint16_t*>(h_d);
  a->q_w = q_w_d;
  a->k_w = k_w_d;
  a->partials = reinterpret_cast<float4*>(partials_d);
  a->status = status_d;
  return ENGRAM_OK;
}

size_t project8_smem_bytes(bool pair) {
  return (pair ? 1024 + STAGES82 * (STAGE82_BYTES + SF_BYTES) : 1024 + STAGES8 * (STAGE8_BYTES + SF_BYTES)) +
         sizeof(SmemCtl) + 16 + sizeof(Comb8);
}

int launch8(bool pair, bool fused, const CUtensorMap* tm, const ProjArgs& a, cudaStream_t st) {
  const void* fn = pair ? (fused ? reinterpret_cast<const void*>(&project82_kernel<true>)
                                 : reinterpret_cast<const void*>(&project82_kernel<false>))
                        : (fused ? reinterpret_cast<const void*>(&project8_kernel<true>)
                                 : reinterpret_cast<const void*>(&project8_kernel<false>));
  const size_t smem = project8_smem_bytes(pair);
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaFuncSetAttribute(project8): %s", cudaGetErrorString(err));
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  cudaLaunchConfig_t cfg = {};
  const int threads = fused ? kThreads8 : kThreads8u;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  int units = 0;  // CTAs (single) or CTA pairs that can be resident at once
  if (pair) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = 2;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
    cfg.gridDim = dim3(2 * (sms / 2));
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    err = cudaOccupancyMaxActiveClusters(&units, fn, &cfg);
    if (err != cudaSuccess || units < 1)
      return fail(ENGRAM_E_CUDA, "no resident CTA pair for the FP8 projection: %s", cudaGetErrorString(err));
  } else {
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
    if (err != cudaSuccess || per_sm < 1)
      return fail(ENGRAM_E_CUDA, "no resident CTA for the FP8 projection: %s", cudaGetErrorString(err));
    units = sms * per_sm;
  }
  if (fused && use_cooperative()) {
    attr[nattr].id = cudaLaunchAttributeCooperative;
    attr[nattr].val.cooperative = 1;
    ++nattr;
  }
  const int n = a.num_tiles < units ? a.num_tiles : units;
  cfg.gridDim = dim3(pair ? 2 * n : n);
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  if (pair)
    err = fused ? cudaLaunchKernelEx(&cfg, project82_kernel<true>, tm[0], tm[1], tm[2], tm[3], a)
                : cudaLaunchKernelEx(&cfg, project82_kernel<false>, tm[0], tm[1], tm[2], tm[3], a);
  else
    err = fused ? cudaLaunchKernelEx(&cfg, project8_kernel<true>, tm[0], tm[1], tm[2], tm[3], a)
                : cudaLaunchKernelEx(&cfg, project8_kernel<false>, tm[0], tm[1], tm[2], tm[3], a);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "project8 kernel launch: %s", cudaGetErrorString(err));
  return check_launch("project8 kernel");
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" int engram_pack_wkv(const uint16_t* wkv_d, int64_t K, int64_t N, uint16_t* wkv_packed_d,
                               void* stream) {
  if (K < 1 || N < 1) return fail(ENGRAM_E_INVALID, "K and N must be positive");
  if (K % 64 != 0 || N % 128 != 0) return fail(ENGRAM_E_SHAPE, "K must be a multiple of 64 and N of 128");
  if (!wkv_d || !wkv_packed_d) return fail(ENGRAM_E_INVALID, "null device pointer");
  if (wkv_d == wkv_packed_d) return fail(ENGRAM_E_INVALID, "in-place repack is not supported");
  int rc = check_device(nullptr);
  if (rc) return rc;
  const int64_t gx = (N + 31) / 32, gy = (K + 31) / 32;
  if (gy > 65535) return fail(ENGRAM_E_SHAPE, "K too large");
  pack_wkv_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), dim3(32, 8), 0,
                    as_stream(stream)>>>(wkv_d, K, N, wkv_packed_d);
  return check_launch("pack_wkv_kernel");
}

extern "C" size_t engram_project_partials_bytes(int64_t n_tokens, int32_t hidden, int32_t hc) {
  if (n_tokens < 0 || hidden < 256 || hc < 1) return 0;
  return static_cast<size_t>(n_tokens) * hc * (hidden / 256) * 4 * sizeof(float);
}

extern "C" int engram_project(const uint16_t* e_d, int64_t n_tokens, int64_t K,
                              const uint16_t* wkv_packed_d, int32_t hidden, int32_t hc,
                              const uint16_t* h_d, const float* q_w_d, const float* k_w_d,
                              float* partials_d, uint16_t* v_d, int32_t* status_d, void* stream) {
  if (!v_d && n_tokens > 0) return fail(ENGRAM_E_INVALID, "null device pointer");
  if (v_d && !aligned(v_d, 16)) return fail(ENGRAM_E_ALIGN, "v must be 16-byte aligned");
  const bool pair = use_pair_kernel(n_tokens);
  ProjArgs a;
  CUtensorMap tmA, tmB;
  int rc = prepare(e_d, n_tokens, K, wkv_packed_d, hidden, hc, h_d, q_w_d, k_w_d, partials_d, status_d, pair, &a,
                   &tmA, &tmB);
  if (rc || n_tokens == 0) return rc;
  a.v = v_d;
  return launch(pair, false, tmA, tmB, a, as_stream(stream));
}

namespace {
// Fused-mode workspace: [partials | counters: cnt[mt][hc][4], ready[mt], abort | gates[mt*128][hc]],
// each part starting on a 256-byte boundary.
// Up to this many tokens engram_project_gate runs the two-kernel path (the
// projection storing v, then the gate kernel) inside its workspace: at decode
// sizes the whole projection is one or two waves of tiles and the fused
// kernel's key-then-value dependency costs more than the separate gate pass
// (measured on GB300: 256 tokens 114 us fused vs ~99 us two-kernel; break-even
// near 2048 tokens).
constexpr int64_t kTwoKernelMaxTokens = 1536;
// Below this K the bf16 path always runs the two kernels: with few k-blocks per
// tile the fused kernel's value tiles wait on their block's gates and their h
// traffic is not hidden behind the main loop (GB300, 16,384 tokens, hidden
// 2560: K 1280 fused 715 us vs 470 us, K 2560 807 vs 725 us; from K 4096 the
// fused kernel wins, 1027 vs 1090 us, and at K 6144, hidden 5120, 3.05 vs
// 3.29 ms).
constexpr int64_t kFusedMinK = 3200;

// The block-FP8 projection keeps a single accumulator buffer (TMEM also holds
// the scale factors), so its fused epilogue cannot overlap the next tile's
// main loop; the two kernels are faster at every size measured (16,384
// tokens, hidden 5120: projection + gate 2.03 ms vs 2.53 ms fused).
// engram_kernel_options.fp8_fused selects the fused FP8 kernel above 1536
// tokens (for comparisons).
bool use_fp8_fused() { return kernel_options().fp8_fused != 0; }

struct FusedWs {
  size_t partials, counters_off, counter_words, gates_off, v_off, total;
};
FusedWs fused_ws(int64_t n_tokens, int32_t hidden, int32_t hc) {
  FusedWs w;
  // 128-row blocks; the CTA-pair kernel's last 256-row tile may reach one past ceil(M/128)
  const size_t mt = 2 * static_cast<size_t>((n_tokens + 2 * BM - 1) / (2 * BM));
  w.partials = engram_project_partials_bytes(n_tokens, hidden, hc);
  w.counters_off = (w.partials + 255) / 256 * 256;
  w.counter_words = mt * hc * 4 + mt + 1;
  w.gates_off = w.counters_off + (w.counter_words * 4 + 255) / 256 * 256;
  w.v_off = w.gates_off + (mt * BM * hc * sizeof(float) + 255) / 256 * 256;
  w.total = w.v_off + static_cast<size_t>(n_tokens) * hidden * 2;  // v of the two-kernel path
  return w;
}
}  // namespace

extern "C" size_t engram_project_gate_workspace_bytes(int64_t n_tokens, int32_t hidden, int32_t hc) {
  if (n_tokens < 0 || hidden < 256 || hc < 1) return 0;
  return fused_ws(n_tokens, hidden, hc).total;
}

extern "C" int engram_project_gate(const uint16_t* e_d, int64_t n_tokens, int64_t K,
                                   const uint16_t* wkv_packed_d, int32_t hidden, int32_t hc, uint16_t* h_d,
                                   const float* q_w_d, const float* k_w_d, const uint8_t* mask_d, float eps,
                                   float clamp, float score_scale, float* gate_out_d, void* workspace_d,
                                   size_t workspace_bytes, int32_t* status_d, void* stream) {
  if (n_tokens > 0 && workspace_d == nullptr) return fail(ENGRAM_E_INVALID, "null workspace");
  if (workspace_d && !aligned(workspace_d, 256)) return fail(ENGRAM_E_ALIGN, "workspace must be 256-byte aligned");
  const size_t need = engram_project_gate_workspace_bytes(n_tokens, hidden, hc);
  if (n_tokens > 0 && workspace_bytes < need)
    return fail(ENGRAM_E_SHAPE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  if (n_tokens > 0 && (n_tokens <= kTwoKernelMaxTokens || K < kFusedMinK)) {
    const FusedWs ws = fused_ws(n_tokens, hidden, hc);
    unsigned char* base = static_cast<unsigned char*>(workspace_d);
    float* partials_d = reinterpret_cast<float*>(base);
    uint16_t* v_d = reinterpret_cast<uint16_t*>(base + ws.v_off);
    int rc = engram_project(e_d, n_tokens, K, wkv_packed_d, hidden, hc, h_d, q_w_d, k_w_d, partials_d, v_d,
                            status_d, stream);
    if (rc) return rc;
    return engram_gate_add(partials_d, v_d, h_d, mask_d, n_tokens, hidden, hc, eps, clamp, score_scale, gate_out_d,
                           stream);
  }
  const bool pair = use_pair_kernel(n_tokens);
  ProjArgs a;
  CUtensorMap tmA, tmB;
  float* partials_d = static_cast<float*>(workspace_d);
  int rc = prepare(e_d, n_tokens, K, wkv_packed_d, hidden, hc, h_d, q_w_d, k_w_d, partials_d, status_d, pair, &a,
                   &tmA, &tmB);
  if (rc || n_tokens == 0) return rc;
  const FusedWs ws = fused_ws(n_tokens, hidden, hc);
  unsigned char* base = static_cast<unsigned char*>(workspace_d);
  const int mt_ws = 2 * a.mt2;
  a.cnt = reinterpret_cast<int32_t*>(base + ws.counters_off);
  a.ready = a.cnt + static_cast<size_t>(mt_ws) * hc * 4;
  a.abort_g = a.ready + mt_ws;
  a.gates = reinterpret_cast<float*>(base + ws.gates_off);
  a.mask = mask_d;
  a.gate_out = gate_out_d;
  a.eps = eps;
  a.clamp = clamp;
  a.score_scale = score_scale;
  cudaStream_t st = as_stream(stream);
  cudaError_t err = cudaMemsetAsync(a.cnt, 0, ws.counter_words * sizeof(int32_t), st);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaMemsetAsync(counters): %s", cudaGetErrorString(err));
  return launch(pair, true, tmA, tmB, a, st);
}

extern "C" int engram_pack_wkv_fp8(const uint8_t* w8_d, const uint8_t* sf_d, int64_t K, int64_t N,
                                   uint8_t* w8_packed_d, uint32_t* sf_packed_d, void* stream) {
  if (K < 1 || N < 1) return fail(ENGRAM_E_INVALID, "K and N must be positive");
  if (K % 128 != 0 || N % 128 != 0) return fail(ENGRAM_E_SHAPE, "K and N must be multiples of 128");
  if (!w8_d || !sf_d || !w8_packed_d || !sf_packed_d) return fail(ENGRAM_E_INVALID, "null device pointer");
  if (!aligned(sf_packed_d, 4)) return fail(ENGRAM_E_ALIGN, "packed scales must be 4-byte aligned");
  int rc = check_device(nullptr);
  if (rc) return rc;
  const int64_t gx = (N + 31) / 32, gy = (K + 31) / 32;
  if (gy > 65535) return fail(ENGRAM_E_SHAPE, "K too large");
  pack_wkv8_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), dim3(32, 8), 0,
                     as_stream(stream)>>>(w8_d, sf_d, K, N, w8_packed_d, sf_packed_d);
  return check_launch("pack_wkv8_kernel");
}

extern "C" int engram_project_fp8(const uint8_t* e8_d, const uint32_t* sfa_d, int64_t n_tokens, int64_t K,
                                  const uint8_t* w8_packed_d, const uint32_t* sfb_d, int32_t hidden, int32_t hc,
                                  const uint16_t* h_d, const float* q_w_d, const float* k_w_d, float* partials_d,
                                  uint16_t* v_d, int32_t* status_d, void* stream) {
  if (!v_d && n_tokens > 0) return fail(ENGRAM_E_INVALID, "null device pointer");
  if (v_d && !aligned(v_d, 16)) return fail(ENGRAM_E_ALIGN, "v must be 16-byte aligned");
  ProjArgs a;
  CUtensorMap tm[4];
  const bool pair = use_fp8_pair();
  int rc = prepare8(e8_d, sfa_d, n_tokens, K, w8_packed_d, sfb_d, hidden, hc, h_d, q_w_d, k_w_d, partials_d,
                    status_d, pair, &a, tm);
  if (rc || n_tokens == 0) return rc;
  a.v = v_d;
  return launch8(pair, false, tm, a, as_stream(stream));
}

extern "C" int engram_project_gate_fp8(const uint8_t* e8_d, const uint32_t* sfa_d, int64_t n_tokens, int64_t K,
                                       const uint8_t* w8_packed_d, const uint32_t* sfb_d, int32_t hidden, int32_t hc,
                                       uint16_t* h_d, const float* q_w_d, const float* k_w_d, const uint8_t* mask_d,
                                       float eps, float clamp, float score_scale, float* gate_out_d,
                                       void* workspace_d, size_t workspace_bytes, int32_t* status_d, void* stream) {
  if (n_tokens > 0 && workspace_d == nullptr) return fail(ENGRAM_E_INVALID, "null workspace");
  if (workspace_d && !aligned(workspace_d, 256)) return fail(ENGRAM_E_ALIGN, "workspace must be 256-byte aligned");
  const size_t need = engram_project_gate_workspace_bytes(n_tokens, hidden, hc);
  if (n_tokens > 0 && workspace_bytes < need)
    return fail(ENGRAM_E_SHAPE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  const FusedWs ws = fused_ws(n_tokens, hidden, hc);
  unsigned char* base = static_cast<unsigned char*>(workspace_d);
  if (n_tokens > 0 && (n_tokens <= kTwoKernelMaxTokens || !use_fp8_fused())) {
    float* partials_d = reinterpret_cast<float*>(base);
    uint16_t* v_d = reinterpret_cast<uint16_t*>(base + ws.v_off);
    int rc = engram_project_fp8(e8_d, sfa_d, n_tokens, K, w8_packed_d, sfb_d, hidden, hc, h_d, q_w_d, k_w_d,
                                partials_d, v_d, status_d, stream);
    if (rc) return rc;
    return engram_gate_add(partials_d, v_d, h_d, mask_d, n_tokens, hidden, hc, eps, clamp, score_scale, gate_out_d,
                           stream);
  }
  ProjArgs a;
  CUtensorMap tm[4];
  const bool pair = use_fp8_pair();
  int rc = prepare8(e8_d, sfa_d, n_tokens, K, w8_packed_d, sfb_d, hidden, hc, h_d, q_w_d, k_w_d,
                    static_cast<float*>(workspace_d), status_d, pair, &a, tm);
  if (rc || n_tokens == 0) return rc;
  const int mt_ws = 2 * a.mt2;
  a.cnt = reinterpret_cast<int32_t*>(base + ws.counters_off);
  a.ready = a.cnt + static_cast<size_t>(mt_ws) * hc * 4;
  a.abort_g = a.ready + mt_ws;
  a.gates = reinterpret_cast<float*>(base + ws.gates_off);
  a.mask = mask_d;
  a.gate_out = gate_out_d;
  a.eps = eps;
  a.clamp = clamp;
  a.score_scale = score_scale;
  cudaStream_t st = as_stream(stream);
  cudaError_t err = cudaMemsetAsync(a.cnt, 0, ws.counter_words * sizeof(int32_t), st);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaMemsetAsync(counters): %s", cudaGetErrorString(err));
  return launch8(pair, true, tm, a, st);
}

extern "C" int engram_selftest_wait(int32_t which, int32_t* scratch_d, int32_t* status_d, void* stream) {
  if (which != 0 && which != 1) return fail(ENGRAM_E_INVALID, "which must be 0 or 1");
  if (!scratch_d || !status_d) return fail(ENGRAM_E_INVALID, "null device pointer");
  int rc = check_device(nullptr);
  if (rc) return rc;
  cudaStream_t st = as_stream(stream);
  cudaError_t err = cudaMemsetAsync(scratch_d, 0, 2 * sizeof(int32_t), st);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaMemsetAsync(scratch): %s", cudaGetErrorString(err));
  selftest_wait_kernel<<<1, 32, 0, st>>>(which, scratch_d, status_d);
  return check_launch("selftest_wait_kernel");
}
