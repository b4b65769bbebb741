// Stage 4 of the Engram lookup: gather 24 rows of 264 bytes per position and
// dequantise them (E4M3 x E8M0 per 32 elements) to bf16.
//
// Pages cited by title:
//   [P-V41] "DeepSeek-V4.1 模型结构（5）：记忆，Engram" §"196B 参数怎么存、怎么取"
//   [P-DS4] "ds4.c 学习笔记" -- glossary entry "Engram", §布局与哈希探测 and
//           §永不常驻的 I/O 设计 (the e4m3_e8m0_32_row264 row format)
//   [P-O1]  "条件记忆：DeepSeek V4.1 Engram 如何用 O(1) 查表换掉一层计算" §2.3
//
// Design (GB300): the rows are scattered at random over a table of up to
// ~100 GB, so the kernel is bound by HBM latency and bandwidth.  Row r starts
// at byte 264 r, which is 16-byte aligned for even r and 8 bytes past a
// 16-byte boundary for odd r; the 16-byte-aligned 272-byte window that
// starts at or 8 bytes before the row covers it in both cases.  Each warp
// runs its own pipeline of `stages` positions: lanes 0..n_cols-1 each issue
// one 272-byte bulk copy (cp.async.bulk, completion counted on the stage's
// mbarrier) into shared memory, so ~100 rows per SM are in flight.  When a
// stage lands, each lane dequantises 8 consecutive elements of every row in
// registers and the warp writes each 512-byte bf16 row segment with one
// coalesced 16-byte store per lane.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdlib>

#include "engram_internal.h"
#include "hash_device.cuh"

namespace engram {
namespace {

constexpr int kRowBytes = ENGRAM_ROW_BYTES;  // 264
constexpr int kSlot = 272;                   // 16-byte aligned window of a row
// Warps per CTA, each an independent pipeline; shared memory then allows 2
// stages per warp.  16 warps x 2 stages beat 8 x 4 with the same bytes in
// flight (GB300: 0.80 vs 0.72 of HBM on 65,536 tokens, 79 vs 107 us for the
// fused hash + gather in the 16,384-token layer step): the other warps'
// dequantisation hides each warp's wait.
constexpr int kWarps = 16;

struct GatherArgs {
  const uint8_t* table;
  int64_t total_rows;
  int64_t table_bytes;
  const int32_t* rows;
  int64_t n_tokens;
  int32_t n_cols;
  int32_t stages;
  uint16_t* e;
  int32_t* status;
};

// Two E4M3 codes (low byte = first element) -> two bf16 values scaled by
// 2^(s-127).  E4M3 -> f16 is exact, f16 -> f32 is exact, the product by a
// power of two is exact in fp32 for every code and scale (an E4M3 value has
// 4 significant bits and the smallest product, 2^-136, is above fp32's
// subnormal resolution), so the single rounding is the final RNE to bf16.
__device__ __forceinline__ uint32_t dq2(uint32_t two, float scale) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two)));
  __half2 hv = *reinterpret_cast<__half2*>(&h2);
  float2 f = __half22float2(hv);
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<uint32_t*>(&b);
}

// E8M0 scale 2^(s-127) as fp32: s = 0 is the subnormal 2^-127, s = 255 is NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  if (s == 0) return __uint_as_float(0x00400000u);
  if (s == 255) return __uint_as_float(0x7fc00000u);
  return __uint_as_float(s << 23);
}

__device__ __forceinline__ uint4 dequant8(uint2 w, uint32_t sbyte) {
  const float sc = e8m0_to_f32(sbyte);
  uint4 o;
  o.x = dq2(w.x & 0xffffu, sc);
  o.y = dq2(w.x >> 16, sc);
  o.z = dq2(w.y & 0xffffu, sc);
  o.w = dq2(w.y >> 16, sc);
  return o;
}

__global__ void __launch_bounds__(kWarps * 32, 1) gather_dequant_kernel(GatherArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // Launched as a programmatic dependent: nothing is read before the
  // previous kernel has finished, and a following history commit may start
  // (and load its inputs) only after that, never ahead of this kernel's own
  // predecessor.
  wait_prior_grids();
  allow_dependent_launch();
  const int w = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t stage_bytes = static_cast<uint32_t>(a.n_cols) * kSlot;
  const int S = a.stages;
  uint8_t* wbuf = smem + static_cast<size_t>(w) * S * stage_bytes;
  uint8_t* meta = smem + static_cast<size_t>(kWarps) * S * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta) + w * S;
  uint32_t* masks = reinterpret_cast<uint32_t*>(meta + kWarps * S * 8) + w * S * 2;

  if (lane == 0)
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&bars[s]), 1);
  fence_mbar_init();
  __syncwarp();

  // warps numbered CTA-minor, so a small batch (a decode step) spreads over
  // every CTA of the grid rather than filling the first few
  const int64_t gw = static_cast<int64_t>(w) * gridDim.x + blockIdx.x;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
  const int n_cols = a.n_cols;

  // Issue the bulk copies of position t into stage s.
  auto issue = [&](int64_t t, int s) {
    int32_t r = -1;
    bool valid = false;
    if (lane < static_cast<uint32_t>(n_cols)) {
      r = a.rows != nullptr ? __ldg(a.rows + t * n_cols + lane) : static_cast<int32_t>(t * n_cols + lane);
      valid = r >= 0 && static_cast<int64_t>(r) < a.total_rows;
      if (!valid && a.status) atomicOr(a.status, static_cast<int>(ENGRAM_ST_BAD_ROW));
    }
    // An even row's window extends 8 bytes past the row; for the table's last
    // row that may pass the end of the allocation, so such a row copies its
    // 256 weight bytes in bulk and its 8 scale bytes with a plain load.
    const bool tail = valid && !(r & 1) && static_cast<int64_t>(r) * kRowBytes + kSlot > a.table_bytes;
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    const uint32_t odd = __ballot_sync(0xffffffffu, valid && (r & 1));
    const uint32_t tmask = __ballot_sync(0xffffffffu, tail);
    const uint32_t bytes = __popc(vmask & ~tmask) * kSlot + __popc(tmask) * 256u;
    const uint32_t bar = smem_u32(&bars[s]);
    uint8_t* dst = wbuf + static_cast<size_t>(s) * stage_bytes + lane * kSlot;
    if (lane == 0) {
      masks[2 * s] = odd;
      masks[2 * s + 1] = vmask;
      mbar_arrive_expect_tx(bar, bytes);
    }
    __syncwarp();
    if (valid) {
      const int64_t off = static_cast<int64_t>(r) * kRowBytes;
      const uint8_t* src = a.table + (off & ~int64_t(15));
      if (!tail) {
        bulk_g2s(smem_u32(dst), src, kSlot, bar);
      } else {
        bulk_g2s(smem_u32(dst), src, 256, bar);
        *reinterpret_cast<uint2*>(dst + 256) = __ldg(reinterpret_cast<const uint2*>(a.table + off + 256));
      }
    }
  };

  // prologue: fill every stage
  for (int s = 0; s < S; ++s) {
    const int64_t t = gw + s * nw;
    if (t < a.n_tokens) issue(t, s);
  }

  int64_t k = 0;
  bool timed_out = false;
  for (;; ++k) {
    const int64_t t = gw + k * nw;
    if (t >= a.n_tokens) break;
    const int s = static_cast<int>(k % S);
    const uint32_t parity = static_cast<uint32_t>((k / S) & 1);
    if (!mbar_wait_bounded(smem_u32(&bars[s]), parity, nullptr)) {
      timed_out = true;
      break;
    }
    const uint32_t odd = masks[2 * s];
    const uint32_t vm = masks[2 * s + 1];
    const uint8_t* sb = wbuf + static_cast<size_t>(s) * stage_bytes;
    uint16_t* out = a.e + t * static_cast<int64_t>(n_cols) * ENGRAM_HEAD_DIM;
#pragma unroll 4
    for (int j = 0; j < n_cols; ++j) {
      const uint8_t* row = sb + j * kSlot + (((odd >> j) & 1u) ? 8 : 0);
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if ((vm >> j) & 1u) {
        const uint2 wv = *reinterpret_cast<const uint2*>(row + lane * 8);
        const uint32_t sbyte = row[256 + (lane >> 2)];
        o = dequant8(wv, sbyte);
      }
      *reinterpret_cast<uint4*>(out + j * ENGRAM_HEAD_DIM + lane * 8) = o;
    }
    __syncwarp();
    const int64_t t2 = t + static_cast<int64_t>(S) * nw;
    if (t2 < a.n_tokens) {
      fence_proxy_async_smem();  // order this warp's shared reads before the async refill
      issue(t2, s);
    }
  }
  if (timed_out) {
    if (lane == 0 && a.status) atomicOr(a.status, static_cast<int>(ENGRAM_ST_TIMEOUT));
    // Let every copy already issued land before the CTA's shared memory is
    // released: wait (bounded) on each outstanding stage.
    for (int64_t kk = k; kk < k + S; ++kk) {
      const int64_t t = gw + kk * nw;
      if (t >= a.n_tokens) break;
      const int s = static_cast<int>(kk % S);
      mbar_wait_bounded(smem_u32(&bars[s]), static_cast<uint32_t>((kk / S) & 1), nullptr);
    }
  }
}


// 16-byte (or 8-byte) asynchronous global -> shared copies through the L1/LSU
// path; completion of a thread's earlier copies is signalled on an mbarrier.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Where the row ids of a position come from.  A warp takes its positions t0,
// t0 + stride, ... in order; fetch() loads the source words of a batch of
// batch() consecutive ones in one warp load, and operator() turns the words
// into position k's row id of column `lane` (warp-collective).  The kernel
// fetches the next batch while the current one's copies are in flight.
//
// Row ids read from memory (or the identity t * n_cols + j for contiguous
// rows), one position per batch ...
struct IdRows {
  const int32_t* rows;
  __device__ __forceinline__ int batch() const { return 1; }
  __device__ __forceinline__ int32_t fetch(int64_t t0, int64_t, int64_t n_tokens, uint32_t lane, int n_cols) const {
    if (t0 >= n_tokens || lane >= static_cast<uint32_t>(n_cols)) return -1;
    return rows != nullptr ? __ldg(rows + t0 * n_cols + lane) : static_cast<int32_t>(t0 * n_cols + lane);
  }
  __device__ __forceinline__ int32_t operator()(int32_t word, int, int64_t, uint32_t, int) const { return word; }
};

// ... or computed in the warp from the position's token window (the fused
// hash + gather: the row ids need not round-trip through memory; they and
// the mask are still written when asked for).  One fetch loads the window
// slots of 32 / max_ngram positions.
struct HashedRows {
  hashdev::HashConsts c;
  const int32_t* raw;
  const int64_t* cu;
  int32_t n_seqs;
  const int32_t* tmap;
  const int32_t* hist;
  int32_t* rows_out;  // or null
  uint8_t* mask;
  int32_t* status;
  __device__ __forceinline__ int batch() const { return 32 / c.max_ngram; }
  __device__ __forceinline__ int32_t fetch(int64_t t0, int64_t stride, int64_t n_tokens, uint32_t, int) const {
    return hashdev::prefill_slot_batch(c, t0, stride, n_tokens, raw, cu, n_seqs, tmap, hist, status);
  }
  __device__ __forceinline__ int32_t operator()(int32_t word, int k, int64_t t, uint32_t lane, int n_cols) const {
    int32_t row;
    const bool dead = hashdev::window_rows(word, c, &row, k * c.max_ngram);
    if (rows_out != nullptr && lane < static_cast<uint32_t>(n_cols)) rows_out[t * n_cols + lane] = row;
    if (lane == 0) mask[t] = dead ? 1 : 0;
    return row;
  }
};

// ... or computed from a decode entry's new id and its carried history, the
// history rolled in the same warp once every lane has read its slot (entries
// of one call name distinct slots, so no other warp touches it).  Nothing is
// fetched ahead: the entry reads its slot's history when it is issued.
struct StepRows {
  hashdev::HashConsts c;
  const int32_t* raw;
  const int32_t* slots;
  const int32_t* tmap;
  int32_t* hist;
  int64_t n_slots;
  int32_t* rows_out;  // or null
  uint8_t* mask;
  int32_t* status;
  __device__ __forceinline__ int batch() const { return 1; }
  __device__ __forceinline__ int32_t fetch(int64_t, int64_t, int64_t, uint32_t, int) const { return 0; }
  __device__ __forceinline__ int32_t operator()(int32_t, int, int64_t b, uint32_t lane, int n_cols) const {
    bool pad_row;
    int32_t xnew;
    const int32_t slot = hashdev::step_slot(c, b, raw, slots, tmap, hist, n_slots, status, &pad_row, &xnew);
    int32_t row;
    const bool dead = hashdev::window_rows(slot, c, &row);
    if (rows_out != nullptr && lane < static_cast<uint32_t>(n_cols)) rows_out[b * n_cols + lane] = row;
    if (lane == 0) mask[b] = (dead || pad_row) ? 1 : 0;
    __syncwarp();
    hashdev::step_commit(c, b, slots, hist, pad_row, xnew, slot);
    return row;
  }
};

// What a warp writes for a position once its rows sit in shared memory
// (row j at sb + j * 272 + 8 if odd): dequantised bf16 rows ...
struct Bf16Out {
  uint16_t* e;  // [T][n_cols * 256]
  __device__ __forceinline__ void operator()(const uint8_t* sb, uint32_t odd, uint32_t vm, int64_t t, int n_cols,
                                             uint32_t lane) const {
    uint16_t* out = e + t * static_cast<int64_t>(n_cols) * ENGRAM_HEAD_DIM;
#pragma unroll 4
    for (int j = 0; j < n_cols; ++j) {
      const uint8_t* row = sb + j * kSlot + (((odd >> j) & 1u) ? 8 : 0);
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if ((vm >> j) & 1u) {
        const uint2 wv = *reinterpret_cast<const uint2*>(row + lane * 8);
        const uint32_t sbyte = row[256 + (lane >> 2)];
        o = dequant8(wv, sbyte);
      }
      *reinterpret_cast<uint4*>(out + j * ENGRAM_HEAD_DIM + lane * 8) = o;
    }
  }
};

// ... or the rows as they are, for the block-scaled FP8 projection: the E4M3
// bytes concatenated, e8[t][256 j + c], and the E8M0 scales grouped by
// 128-element k-block: row kb = 2 j + b / 4 of sf holds T128 words (T rounded
// up to a multiple of 128), byte b % 4 of position t's word the scale of its
// 32-element block b of row j, positions in sf_word_index order (so a
// k-block's scales of 128 positions form the 512-byte image the projection
// copies to TMEM as it is).  A bad row becomes zero bytes with scale 127 (the
// value 0); positions T .. T128 - 1 hold scale 127 too.
struct Fp8Out {
  uint8_t* e8;    // [T][n_cols * 256]
  uint32_t* sf;   // [n_cols * 2][T128] words of four E8M0 bytes
  int64_t n_tokens;
  __device__ __forceinline__ void operator()(const uint8_t* sb, uint32_t odd, uint32_t vm, int64_t t, int n_cols,
                                             uint32_t lane) const {
    uint8_t* out = e8 + t * static_cast<int64_t>(n_cols) * ENGRAM_HEAD_DIM;
#pragma unroll 4
    for (int j = 0; j < n_cols; ++j) {
      const uint8_t* row = sb + j * kSlot + (((odd >> j) & 1u) ? 8 : 0);
      const uint2 wv = ((vm >> j) & 1u) ? *reinterpret_cast<const uint2*>(row + lane * 8) : make_uint2(0u, 0u);
      *reinterpret_cast<uint2*>(out + j * ENGRAM_HEAD_DIM + lane * 8) = wv;
    }
    if (lane < static_cast<uint32_t>(n_cols)) {
      const int64_t ld = (n_tokens + 127) & ~int64_t(127);
      uint32_t* s0 = sf + 2 * static_cast<int64_t>(lane) * ld;
      const uint8_t* row = sb + lane * kSlot + (((odd >> lane) & 1u) ? 8 : 0);
      const uint2 sc = ((vm >> lane) & 1u) ? *reinterpret_cast<const uint2*>(row + 256) : make_uint2(0x7f7f7f7fu, 0x7f7f7f7fu);
      s0[sf_word_index(t)] = sc.x;
      s0[ld + sf_word_index(t)] = sc.y;
      if (t == n_tokens - 1)  // the last position also fills the padding of its 128-block
        for (int64_t p = n_tokens; p < ld; ++p) {
          s0[sf_word_index(p)] = 0x7f7f7f7fu;
          s0[ld + sf_word_index(p)] = 0x7f7f7f7fu;
        }
    }
  }
};

// Same pipeline as gather_dequant_kernel, but each row window moves as 17
// 16-byte cp.async copies spread over the warp's lanes (a flat list of
// n_cols * 17 pieces per position) instead of one bulk copy per row: many
// small requests go through the LSU rather than the TMA unit.
template <class RowSource, class Out>
__global__ void __launch_bounds__(kWarps * 32, 1) gather_ldgsts_kernel(GatherArgs a, RowSource src, Out store) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // Launched as a programmatic dependent: nothing is read before the
  // previous kernel has finished, and a following history commit may start
  // (and load its inputs) only after that, never ahead of this kernel's own
  // predecessor.
  wait_prior_grids();
  allow_dependent_launch();
  const int w = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t stage_bytes = static_cast<uint32_t>(a.n_cols) * kSlot;
  const int S = a.stages;
  uint8_t* wbuf = smem + static_cast<size_t>(w) * S * stage_bytes;
  uint8_t* meta = smem + static_cast<size_t>(kWarps) * S * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta) + w * S;
  uint32_t* masks = reinterpret_cast<uint32_t*>(meta + kWarps * S * 8) + w * S * 2;

  if (lane == 0)
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&bars[s]), 32);  // one async arrival per lane
  fence_mbar_init();
  __syncwarp();

  // warps numbered CTA-minor, so a small batch (a decode step) spreads over
  // every CTA of the grid rather than filling the first few
  const int64_t gw = static_cast<int64_t>(w) * gridDim.x + blockIdx.x;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
  const int n_cols = a.n_cols;
  const int pieces = n_cols * 17;

  // the source words of the batch holding the next position to issue, and
  // of the batch after it (fetched once that batch's first copies are out)
  const int B = src.batch();
  int64_t qb = 0;  // the current batch's first position, counted per warp
  int32_t cur = src.fetch(gw, nw, a.n_tokens, lane, n_cols);
  int32_t nxt = 0;

  // issues the copies of the warp's position q (t = gw + q * nw) into stage s
  auto issue = [&](int64_t q, int s) {
    if (q == qb + B) {
      cur = nxt;
      qb += B;
    }
    const int64_t t = gw + q * nw;
    const int32_t r = src(cur, static_cast<int>(q - qb), t, lane, n_cols);  // warp-collective
    bool valid = false;
    if (lane < static_cast<uint32_t>(n_cols)) {
      valid = r >= 0 && static_cast<int64_t>(r) < a.total_rows;
      if (!valid && a.status) atomicOr(a.status, static_cast<int>(ENGRAM_ST_BAD_ROW));
    }
    // an even row whose 272-byte window passes the end of the allocation
    // copies its last piece as the 8 scale bytes only
    const bool tail = valid && !(r & 1) && static_cast<int64_t>(r) * kRowBytes + kSlot > a.table_bytes;
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    const uint32_t odd = __ballot_sync(0xffffffffu, valid && (r & 1));
    const uint32_t tmask = __ballot_sync(0xffffffffu, tail);
    if (lane == 0) {
      masks[2 * s] = odd;
      masks[2 * s + 1] = vmask;
    }
    const uint32_t sbase = smem_u32(wbuf + static_cast<size_t>(s) * stage_bytes);
    for (int p0 = 0; p0 < pieces; p0 += 32) {
      const int p = p0 + static_cast<int>(lane);
      const int row = p / 17;
      const int piece = p - 17 * row;
      const int rr = __shfl_sync(0xffffffffu, r, row < 32 ? row : 0);
      if (p < pieces && ((vmask >> row) & 1u)) {
        const uint8_t* from = a.table + ((static_cast<int64_t>(rr) * kRowBytes) & ~int64_t(15)) + piece * 16;
        const uint32_t dst = sbase + row * kSlot + piece * 16;
        if (piece == 16 && ((tmask >> row) & 1u)) cp_async8(dst, from);
        else cp_async16(dst, from);
      }
    }
    cp_async_arrive(smem_u32(&bars[s]));
    if (q == qb) nxt = src.fetch(gw + (qb + B) * nw, nw, a.n_tokens, lane, n_cols);
  };

  for (int s = 0; s < S; ++s)
    if (gw + s * nw < a.n_tokens) issue(s, s);

  int64_t k = 0;
  bool timed_out = false;
  for (;; ++k) {
    const int64_t t = gw + k * nw;
    if (t >= a.n_tokens) break;
    const int s = static_cast<int>(k % S);
    const uint32_t parity = static_cast<uint32_t>((k / S) & 1);
    if (!mbar_wait_bounded(smem_u32(&bars[s]), parity, nullptr)) {
      timed_out = true;
      break;
    }
    store(wbuf + static_cast<size_t>(s) * stage_bytes, masks[2 * s], masks[2 * s + 1], t, n_cols, lane);
    __syncwarp();
    if (t + static_cast<int64_t>(S) * nw < a.n_tokens) issue(k + S, s);
  }
  if (timed_out) {
    if (lane == 0 && a.status) atomicOr(a.status, static_cast<int>(ENGRAM_ST_TIMEOUT));
    asm volatile("cp.async.wait_all;" ::: "memory");  // this thread's copies land before exit
  }
}

__global__ void fill_table_kernel(uint8_t* table, int64_t n_words, uint64_t seed) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t wi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; wi < n_words;
       wi += stride) {
    uint64_t v = splitmix64_at(seed, static_cast<uint64_t>(wi));
    if (wi % (kRowBytes / 8) < 32) {
      // weight bytes: an E4M3 NaN code (low 7 bits all ones) becomes byte ^ 1;
      // adding 1 to each byte's low 7 bits sets its bit 7 exactly for 0x7F.
      const uint64_t low7 = v & 0x7F7F7F7F7F7F7F7Full;
      const uint64_t hit = ((low7 + 0x0101010101010101ull) & 0x8080808080808080ull) >> 7;
      v ^= hit;
    } else {
      uint64_t o = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uint64_t byte = (v >> (8 * b)) & 0xFF;
        o |= (120 + byte % 11) << (8 * b);
      }
      v = o;
    }
    reinterpret_cast<uint64_t*>(table)[wi] = v;
  }
}

// The cp.async row copies are the default; engram_kernel_options.gather_copy
// = 1 selects one bulk (TMA) copy per row instead.  Both measure the same on
// GB300.
bool use_ldgsts() { return kernel_options().gather_copy == 0; }

}  // namespace
}  // namespace engram

using namespace engram;

namespace engram {
namespace {

// Pipeline depth and shared memory of the gather kernels for n_cols rows per
// position; launches the cp.async kernel with the given row source.
int gather_config(int n_cols, int* stages, size_t* smem) {
  const int smem_max = 227 * 1024;
  const int per_stage = n_cols * kSlot + 16;  // slots + mbarrier + two masks
  int s = smem_max / (kWarps * per_stage);
  if (s > 4) s = 4;
  if (s < 1) return fail(ENGRAM_E_SHAPE, "n_cols %d does not fit shared memory", n_cols);
  *stages = s;
  *smem = static_cast<size_t>(kWarps) * s * per_stage;
  return ENGRAM_OK;
}

template <class RowSource, class Out>
int launch_ldgsts(const GatherArgs& a, const RowSource& src, const Out& out, size_t smem, int sms, cudaStream_t st) {
  cudaError_t err = cudaFuncSetAttribute(gather_ldgsts_kernel<RowSource, Out>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "cudaFuncSetAttribute(gather): %s", cudaGetErrorString(err));
  // one CTA per SM, or one per position when there are fewer positions
  const int blocks = static_cast<int>(a.n_tokens < sms ? a.n_tokens : sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the launch overlaps the previous kernel's tail
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, gather_ldgsts_kernel<RowSource, Out>, a, src, out);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "gather_ldgsts_kernel launch: %s", cudaGetErrorString(err));
  return check_launch("gather_ldgsts_kernel");
}

}  // namespace
}  // namespace engram

extern "C" int engram_gather_dequant(const uint8_t* table_d, int64_t total_rows,
                                     int64_t table_bytes, const int32_t* row_ids_d,
                                     int64_t n_tokens, int32_t n_cols, uint16_t* e_d,
                                     int32_t* status_d, void* stream) {
  if (n_tokens < 0 || total_rows < 0) return fail(ENGRAM_E_INVALID, "negative size");
  if (n_cols < 1 || n_cols > ENGRAM_MAX_COLS) return fail(ENGRAM_E_SHAPE, "n_cols %d", n_cols);
  if (table_bytes < total_rows * kRowBytes)
    return fail(ENGRAM_E_SHAPE, "table_bytes %lld < total_rows * 264", (long long)table_bytes);
  if (n_tokens == 0) return ENGRAM_OK;
  if (!table_d || !e_d) return fail(ENGRAM_E_INVALID, "null device pointer");  // row_ids_d NULL: identity ids
  if (!aligned(table_d, 16) || !aligned(e_d, 16))
    return fail(ENGRAM_E_ALIGN, "table and e must be 16-byte aligned");
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  int stages = 0;
  size_t smem = 0;
  if ((rc = gather_config(n_cols, &stages, &smem))) return rc;
  GatherArgs a{table_d, total_rows, table_bytes, row_ids_d, n_tokens, n_cols, stages, e_d, status_d};
  if (use_ldgsts()) return launch_ldgsts(a, IdRows{row_ids_d}, Bf16Out{e_d}, smem, sms, as_stream(stream));
  cudaError_t err = cudaFuncSetAttribute(gather_dequant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
  if (err != cudaSuccess)
    return fail(ENGRAM_E_CUDA, "cudaFuncSetAttribute(gather): %s", cudaGetErrorString(err));
  const int blocks = static_cast<int>(n_tokens < sms ? n_tokens : sms);
  gather_dequant_kernel<<<blocks, kWarps * 32, smem, as_stream(stream)>>>(a);
  return check_launch("gather_dequant_kernel");
}

extern "C" int engram_hash_gather(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                                  int64_t n_tokens, const int64_t* cu_seqlens_d, int32_t n_seqs,
                                  const int32_t* token_map_d, int64_t vocab_raw, int32_t* hist_d,
                                  const uint8_t* table_d, int64_t table_bytes, uint16_t* e_d, uint8_t* mask_d,
                                  int32_t* row_ids_d, int32_t* status_d, void* stream) {
  hashdev::HashConsts c;
  int rc = hashdev::make_consts(layout, layer, vocab_raw, &c);
  if (rc) return rc;
  const int64_t total_rows = layout->total_rows[layer];
  if (n_tokens < 0 || n_seqs < 1) return fail(ENGRAM_E_INVALID, "n_tokens < 0 or n_seqs < 1");
  if (table_bytes < total_rows * kRowBytes)
    return fail(ENGRAM_E_SHAPE, "table_bytes %lld < total_rows * 264", (long long)table_bytes);
  if (n_tokens == 0 && hist_d == nullptr) return ENGRAM_OK;
  if (!cu_seqlens_d || !token_map_d || (n_tokens > 0 && (!raw_ids_d || !table_d || !e_d || !mask_d)))
    return fail(ENGRAM_E_INVALID, "null device pointer");
  if (n_tokens > 0 && (!aligned(table_d, 16) || !aligned(e_d, 16)))
    return fail(ENGRAM_E_ALIGN, "table and e must be 16-byte aligned");
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  cudaStream_t st = as_stream(stream);
  if (n_tokens > 0) {
    int stages = 0;
    size_t smem = 0;
    if ((rc = gather_config(c.n_cols, &stages, &smem))) return rc;
    GatherArgs a{table_d, total_rows, table_bytes, nullptr, n_tokens, c.n_cols, stages, e_d, status_d};
    HashedRows src{c, raw_ids_d, cu_seqlens_d, n_seqs, token_map_d, hist_d, row_ids_d, mask_d, status_d};
    if ((rc = launch_ldgsts(a, src, Bf16Out{e_d}, smem, sms, st))) return rc;
  }
  // the history advances after every position has read the old one
  if (hist_d != nullptr)
    return hashdev::launch_hist_commit(c, raw_ids_d, cu_seqlens_d, n_seqs, token_map_d, hist_d, status_d, st);
  return ENGRAM_OK;
}

extern "C" int engram_gather_fp8(const uint8_t* table_d, int64_t total_rows, int64_t table_bytes,
                                 const int32_t* row_ids_d, int64_t n_tokens, int32_t n_cols, uint8_t* e8_d,
                                 uint32_t* sf_d, int32_t* status_d, void* stream) {
  if (n_tokens < 0 || total_rows < 0) return fail(ENGRAM_E_INVALID, "negative size");
  if (n_cols < 1 || n_cols > ENGRAM_MAX_COLS) return fail(ENGRAM_E_SHAPE, "n_cols %d", n_cols);
  if (table_bytes < total_rows * kRowBytes)
    return fail(ENGRAM_E_SHAPE, "table_bytes %lld < total_rows * 264", (long long)table_bytes);
  if (n_tokens == 0) return ENGRAM_OK;
  if (!table_d || !e8_d || !sf_d || !row_ids_d) return fail(ENGRAM_E_INVALID, "null device pointer");
  if (!aligned(table_d, 16) || !aligned(e8_d, 16) || !aligned(sf_d, 16))
    return fail(ENGRAM_E_ALIGN, "table, e8 and sf must be 16-byte aligned");
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  int stages = 0;
  size_t smem = 0;
  if ((rc = gather_config(n_cols, &stages, &smem))) return rc;
  GatherArgs a{table_d, total_rows, table_bytes, row_ids_d, n_tokens, n_cols, stages, nullptr, status_d};
  return launch_ldgsts(a, IdRows{row_ids_d}, Fp8Out{e8_d, sf_d, n_tokens}, smem, sms, as_stream(stream));
}

extern "C" int engram_hash_gather_fp8(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                                      int64_t n_tokens, const int64_t* cu_seqlens_d, int32_t n_seqs,
                                      const int32_t* token_map_d, int64_t vocab_raw, int32_t* hist_d,
                                      const uint8_t* table_d, int64_t table_bytes, uint8_t* e8_d, uint32_t* sf_d,
                                      uint8_t* mask_d, int32_t* row_ids_d, int32_t* status_d, void* stream) {
  hashdev::HashConsts c;
  int rc = hashdev::make_consts(layout, layer, vocab_raw, &c);
  if (rc) return rc;
  const int64_t total_rows = layout->total_rows[layer];
  if (n_tokens < 0 || n_seqs < 1) return fail(ENGRAM_E_INVALID, "n_tokens < 0 or n_seqs < 1");
  if (table_bytes < total_rows * kRowBytes)
    return fail(ENGRAM_E_SHAPE, "table_bytes %lld < total_rows * 264", (long long)table_bytes);
  if (n_tokens == 0 && hist_d == nullptr) return ENGRAM_OK;
  if (!cu_seqlens_d || !token_map_d || (n_tokens > 0 && (!raw_ids_d || !table_d || !e8_d || !sf_d || !mask_d)))
    return fail(ENGRAM_E_INVALID, "null device pointer");
  if (n_tokens > 0 && (!aligned(table_d, 16) || !aligned(e8_d, 16) || !aligned(sf_d, 16)))
    return fail(ENGRAM_E_ALIGN, "table, e8 and sf must be 16-byte aligned");
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  cudaStream_t st = as_stream(stream);
  if (n_tokens > 0) {
    int stages = 0;
    size_t smem = 0;
    if ((rc = gather_config(c.n_cols, &stages, &smem))) return rc;
    GatherArgs a{table_d, total_rows, table_bytes, nullptr, n_tokens, c.n_cols, stages, nullptr, status_d};
    HashedRows src{c, raw_ids_d, cu_seqlens_d, n_seqs, token_map_d, hist_d, row_ids_d, mask_d, status_d};
    if ((rc = launch_ldgsts(a, src, Fp8Out{e8_d, sf_d, n_tokens}, smem, sms, st))) return rc;
  }
  if (hist_d != nullptr)
    return hashdev::launch_hist_commit(c, raw_ids_d, cu_seqlens_d, n_seqs, token_map_d, hist_d, status_d, st);
  return ENGRAM_OK;
}

namespace {
// Shared checks and launch of the fused decode steps (bf16 or FP8 outputs).
template <class Out>
int hash_gather_step(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d, const int32_t* slots_d,
                     int32_t batch, const int32_t* token_map_d, int64_t vocab_raw, int32_t* hist_d, int64_t n_slots,
                     const uint8_t* table_d, int64_t table_bytes, void* out_d, uint8_t* mask_d, int32_t* row_ids_d,
                     int32_t* status_d, void* stream, Out out) {
  hashdev::HashConsts c;
  int rc = hashdev::make_consts(layout, layer, vocab_raw, &c);
  if (rc) return rc;
  const int64_t total_rows = layout->total_rows[layer];
  if (batch < 0 || n_slots < 0) return fail(ENGRAM_E_INVALID, "negative batch or n_slots");
  if (table_bytes < total_rows * kRowBytes)
    return fail(ENGRAM_E_SHAPE, "table_bytes %lld < total_rows * 264", (long long)table_bytes);
  if (batch == 0) return ENGRAM_OK;
  if (!raw_ids_d || !slots_d || !token_map_d || !table_d || !out_d || !mask_d || (n_slots > 0 && !hist_d))
    return fail(ENGRAM_E_INVALID, "null device pointer");
  if (!aligned(table_d, 16) || !aligned(out_d, 16)) return fail(ENGRAM_E_ALIGN, "table and e must be 16-byte aligned");
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  int stages = 0;
  size_t smem = 0;
  if ((rc = gather_config(c.n_cols, &stages, &smem))) return rc;
  GatherArgs a{table_d, total_rows, table_bytes, nullptr, batch, c.n_cols, stages, nullptr, status_d};
  StepRows src{c, raw_ids_d, slots_d, token_map_d, hist_d, n_slots, row_ids_d, mask_d, status_d};
  return launch_ldgsts(a, src, out, smem, sms, as_stream(stream));
}
}  // namespace

extern "C" int engram_hash_gather_step(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                                       const int32_t* slots_d, int32_t batch, const int32_t* token_map_d,
                                       int64_t vocab_raw, int32_t* hist_d, int64_t n_slots, const uint8_t* table_d,
                                       int64_t table_bytes, uint16_t* e_d, uint8_t* mask_d, int32_t* row_ids_d,
                                       int32_t* status_d, void* stream) {
  return hash_gather_step(layout, layer, raw_ids_d, slots_d, batch, token_map_d, vocab_raw, hist_d, n_slots, table_d,
                          table_bytes, e_d, mask_d, row_ids_d, status_d, stream, Bf16Out{e_d});
}

extern "C" int engram_hash_gather_step_fp8(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                                           const int32_t* slots_d, int32_t batch, const int32_t* token_map_d,
                                           int64_t vocab_raw, int32_t* hist_d, int64_t n_slots,
                                           const uint8_t* table_d, int64_t table_bytes, uint8_t* e8_d,
                                           uint32_t* sf_d, uint8_t* mask_d, int32_t* row_ids_d, int32_t* status_d,
                                           void* stream) {
  if (batch > 0 && (sf_d == nullptr || !aligned(sf_d, 16)))
    return fail(ENGRAM_E_INVALID, "sf must be a 16-byte aligned device pointer");
  return hash_gather_step(layout, layer, raw_ids_d, slots_d, batch, token_map_d, vocab_raw, hist_d, n_slots, table_d,
                          table_bytes, e8_d, mask_d, row_ids_d, status_d, stream, Fp8Out{e8_d, sf_d, batch});
}

extern "C" int engram_dequant_rows(const uint8_t* rows_d, int64_t n_rows, int64_t rows_bytes, int32_t n_cols,
                                  uint16_t* e_d, int32_t* status_d, void* stream) {
  if (n_cols < 1 || n_cols > ENGRAM_MAX_COLS) return fail(ENGRAM_E_SHAPE, "n_cols %d", n_cols);
  if (n_rows < 0 || n_rows % n_cols != 0) return fail(ENGRAM_E_SHAPE, "n_rows must be a multiple of n_cols");
  if (n_rows >= (int64_t(1) << 31)) return fail(ENGRAM_E_RANGE, "too many rows");
  // the gather kernel with row ids t*n_cols + j over the contiguous rows
  return engram_gather_dequant(rows_d, n_rows, rows_bytes, nullptr, n_rows / n_cols, n_cols, e_d, status_d, stream);
}

extern "C" int engram_fill_synthetic_table(uint8_t* table_d, int64_t n_rows, uint64_t seed,
                                           void* stream) {
  if (n_rows < 0) return fail(ENGRAM_E_INVALID, "n_rows < 0");
  if (n_rows == 0) return ENGRAM_OK;
  if (!table_d) return fail(ENGRAM_E_INVALID, "null table");
  if (!aligned(table_d, 8)) return fail(ENGRAM_E_ALIGN, "table must be 8-byte aligned");
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  const int64_t n_words = n_rows * (kRowBytes / 8);
  fill_table_kernel<<<sms * 8, 256, 0, as_stream(stream)>>>(table_d, n_words, seed);
  return check_launch("fill_table_kernel");
}
