// Stages 1-3 of the Engram lookup as device helpers shared by the hash
// kernels and the fused hash + gather kernel: the per-layer constants, the
// token map with DEAD handling, the suffix window with pad / carried history,
// the DEAD cascade, the multiplicative-XOR mix and the Barrett modulo.
//
// Pages cited by title:
//   [P-V41]    "DeepSeek-V4.1 模型结构（5）：记忆，Engram" §哈希函数 eq. (H), §一层只有一张表
//   [P-LMNT]   "Engram条件记忆：DeepSeek-V4.1-Flash中196B稀疏参数N-gram哈希查表的实现原理" §多模态细节
//   [P-DS4]    "ds4.c 学习笔记" -- glossary entry "Engram", §布局与哈希探测 step 3
//   [P-DETAIL] "DeepSeek Engram 详解：把静态知识从计算里拆出来" §3.2
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "engram_internal.h"

namespace engram {
namespace hashdev {

constexpr int kDead = ENGRAM_DEAD;

struct HashConsts {
  uint64_t mult[ENGRAM_MAX_NGRAM];
  uint64_t recip[ENGRAM_MAX_COLS];
  uint32_t prime[ENGRAM_MAX_COLS];
  uint32_t offset[ENGRAM_MAX_COLS];
  int32_t n_cols;
  int32_t n_heads;
  int32_t max_ngram;
  int32_t pad_id;
  int64_t vocab;      // V (compressed)
  int64_t vocab_raw;  // V_raw
};

inline int make_consts(const engram_layout* L, int layer, int64_t vocab_raw, HashConsts* c) {
  if (L == nullptr) return fail(ENGRAM_E_INVALID, "null layout");
  if (layer < 0 || layer >= L->n_layers)
    return fail(ENGRAM_E_INVALID, "layer %d not in [0, %d)", layer, L->n_layers);
  if (L->n_cols < 1 || L->n_cols > ENGRAM_MAX_COLS || L->max_ngram < 2 ||
      L->max_ngram > ENGRAM_MAX_NGRAM || L->n_cols != (L->max_ngram - 1) * L->n_heads)
    return fail(ENGRAM_E_SHAPE, "layout has inconsistent column counts");
  if (vocab_raw < 1 || vocab_raw > INT32_MAX) return fail(ENGRAM_E_INVALID, "bad vocab_raw");
  for (int j = 0; j < L->n_cols; ++j) {
    int64_t p = L->primes[layer][j];
    int64_t o = L->offsets[layer][j];
    if (p < 2 || p >= (int64_t(1) << 31) || o < 0 || o + p > (int64_t(1) << 31))
      return fail(ENGRAM_E_RANGE, "column %d prime/offset out of the int32 row range", j);
    c->prime[j] = static_cast<uint32_t>(p);
    c->offset[j] = static_cast<uint32_t>(o);
    c->recip[j] = ~0ull / static_cast<uint64_t>(p);  // recomputed: never trust a stale field
  }
  for (int i = 0; i < L->max_ngram; ++i) c->mult[i] = static_cast<uint64_t>(L->multipliers[layer][i]);
  c->n_cols = L->n_cols;
  c->n_heads = L->n_heads;
  c->max_ngram = L->max_ngram;
  c->pad_id = L->pad_id;
  c->vocab = L->vocab_compressed;
  c->vocab_raw = vocab_raw;
  return ENGRAM_OK;
}

// x mod p for any 64-bit x, with r = floor((2^64-1)/p) precomputed (Barrett
// reduction, Barrett 1986).  q = floor(x r / 2^64) is floor(x/p) or one less,
// so a single conditional subtraction finishes.
__device__ __forceinline__ uint32_t mod_prime(uint64_t x, uint32_t p, uint64_t r) {
  uint64_t q = __umul64hi(x, r);
  uint64_t rem = x - q * static_cast<uint64_t>(p);
  if (rem >= p) rem -= p;
  return static_cast<uint32_t>(rem);
}

// Compressed id of one raw id, DEAD for an image position; an invalid raw id
// or map value reports ENGRAM_ST_BAD_TOKEN and becomes DEAD (masked).
__device__ __forceinline__ int32_t compress_id(int32_t raw, const int32_t* __restrict__ tmap,
                                               const HashConsts& c, int32_t* status) {
  if (raw == kDead) return kDead;
  if (raw < 0 || static_cast<int64_t>(raw) >= c.vocab_raw) {
    if (status) atomicOr(status, static_cast<int>(ENGRAM_ST_BAD_TOKEN));
    return kDead;
  }
  int32_t x = __ldg(tmap + raw);
  if (x < 0 || static_cast<int64_t>(x) >= c.vocab) {
    if (status) atomicOr(status, static_cast<int>(ENGRAM_ST_BAD_TOKEN));
    return kDead;
  }
  return x;
}

// A history entry must be DEAD or a compressed id.
__device__ __forceinline__ int32_t check_hist(int32_t x, const HashConsts& c, int32_t* status) {
  if (x == kDead) return kDead;
  if (x < 0 || static_cast<int64_t>(x) >= c.vocab) {
    if (status) atomicOr(status, static_cast<int>(ENGRAM_ST_BAD_TOKEN));
    return kDead;
  }
  return x;
}

// Given the window slot held by lane base + i, i < max_ngram (slot i =
// x'_{t-i}), applies the DEAD cascade and forms the mixes; lane j < n_cols
// gets the row id of column j (other lanes -1).  Returns whether the position
// itself is DEAD.  All 32 lanes call it.
__device__ __forceinline__ bool window_rows(int32_t my_slot, const HashConsts& c, int32_t* row, int base = 0) {
  const uint32_t lane = lane_id();
  // [P-V41] image tokens / [P-LMNT] §多模态细节: looking back, the first DEAD
  // slot and every slot farther back count as pad.
  uint64_t g[ENGRAM_MAX_NGRAM];
  bool dead_seen = false;
  bool self_dead = false;
#pragma unroll
  for (int i = 0; i < ENGRAM_MAX_NGRAM; ++i) {
    int32_t v = __shfl_sync(0xffffffffu, my_slot, (base + i) & 31);
    if (i < c.max_ngram) {
      if (v == kDead) {
        dead_seen = true;
        if (i == 0) self_dead = true;
      }
      g[i] = static_cast<uint64_t>(dead_seen ? c.pad_id : v);
    } else {
      g[i] = 0;
    }
  }
  *row = -1;
  if (lane < static_cast<uint32_t>(c.n_cols)) {
    // [P-V41] eq. (H): mix_n = XOR_{i<n} x'_{t-i} * m_i; column j is order
    // n = 2 + j / n_heads ([P-DS4] step 3: row = mix mod p + offset).
    const int n = 2 + static_cast<int>(lane) / c.n_heads;
    uint64_t mix = 0;
#pragma unroll
    for (int i = 0; i < ENGRAM_MAX_NGRAM; ++i)
      if (i < n) mix ^= g[i] * c.mult[i];
    const uint32_t z = mod_prime(mix, c.prime[lane], c.recip[lane]);
    *row = static_cast<int32_t>(z + c.offset[lane]);
  }
  return self_dead;
}

// Row ids of one position written out: 24 lanes store 96 bytes, lane 0 the mask.
__device__ __forceinline__ void hash_window(int32_t my_slot, const HashConsts& c,
                                            int32_t* __restrict__ rows_out, uint8_t* mask_out,
                                            bool force_mask) {
  int32_t row;
  const bool self_dead = window_rows(my_slot, c, &row);
  const uint32_t lane = lane_id();
  if (lane < static_cast<uint32_t>(c.n_cols)) rows_out[lane] = row;
  if (lane == 0) *mask_out = (self_dead || force_mask) ? 1 : 0;
}

// Window slot i of prefill position t of packed sequences: x'_{t-i}, or the
// carried history (most recent first) / pad before the sequence start.  Any
// lane may ask for any (t, i).
__device__ __forceinline__ int32_t prefill_slot_at(const HashConsts& c, int64_t t, int i,
                                                   const int32_t* __restrict__ raw, const int64_t* __restrict__ cu,
                                                   int32_t n_seqs, const int32_t* __restrict__ tmap,
                                                   const int32_t* __restrict__ hist, int32_t* status) {
  const int depth = c.max_ngram - 1;
  // sequence of position t: largest s with cu[s] <= t
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int64_t start = __ldg(cu + lo);
  const int64_t src = t - static_cast<int64_t>(i);
  if (src >= start) return compress_id(__ldg(raw + src), tmap, c, status);
  if (hist != nullptr) {
    const int64_t hidx = static_cast<int64_t>(i) - 1 - (t - start);
    return check_hist(__ldg(hist + static_cast<int64_t>(lo) * depth + hidx), c, status);
  }
  return c.pad_id;
}

// The window slot of lane i < max_ngram for prefill position t (other lanes
// return pad).
__device__ __forceinline__ int32_t prefill_slot(const HashConsts& c, int64_t t, const int32_t* __restrict__ raw,
                                                const int64_t* __restrict__ cu, int32_t n_seqs,
                                                const int32_t* __restrict__ tmap, const int32_t* __restrict__ hist,
                                                int32_t* status) {
  const uint32_t lane = lane_id();
  if (lane >= static_cast<uint32_t>(c.max_ngram)) return c.pad_id;
  return prefill_slot_at(c, t, static_cast<int>(lane), raw, cu, n_seqs, tmap, hist, status);
}

// The window slots of a batch of prefill positions t0 + k * stride, k <
// 32 / max_ngram, in one warp load: lane k * max_ngram + i holds slot i of
// position k (pad past n_tokens and on the lanes left over).  window_rows
// with base k * max_ngram then forms position k's row ids.
__device__ __forceinline__ int32_t prefill_slot_batch(const HashConsts& c, int64_t t0, int64_t stride,
                                                      int64_t n_tokens, const int32_t* __restrict__ raw,
                                                      const int64_t* __restrict__ cu, int32_t n_seqs,
                                                      const int32_t* __restrict__ tmap,
                                                      const int32_t* __restrict__ hist, int32_t* status) {
  const int lane = static_cast<int>(lane_id());
  const int k = lane / c.max_ngram;
  const int i = lane - k * c.max_ngram;
  const int64_t t = t0 + static_cast<int64_t>(k) * stride;
  if (k >= 32 / c.max_ngram || t >= n_tokens) return c.pad_id;
  return prefill_slot_at(c, t, i, raw, cu, n_seqs, tmap, hist, status);
}

// The window slot of lane i < max_ngram for decode entry b: lane 0 the new
// compressed id, lanes 1.. the entry's carried history (most recent first),
// all pad for a padding entry (slot < 0) or a slot >= n_slots (which also
// sets ENGRAM_ST_BAD_SLOT).  *pad_row tells the caller the entry commits
// nothing; *xnew (lane 0) is the new id.
__device__ __forceinline__ int32_t step_slot(const HashConsts& c, int64_t b, const int32_t* __restrict__ raw,
                                             const int32_t* __restrict__ slots, const int32_t* __restrict__ tmap,
                                             const int32_t* hist, int64_t n_slots, int32_t* status, bool* pad_row,
                                             int32_t* xnew) {
  const uint32_t lane = lane_id();
  const int depth = c.max_ngram - 1;
  const int32_t sl = slots[b];
  bool pad = sl < 0;
  if (sl >= 0 && static_cast<int64_t>(sl) >= n_slots) {
    if (lane == 0 && status) atomicOr(status, static_cast<int>(ENGRAM_ST_BAD_SLOT));
    pad = true;
  }
  int32_t slot = c.pad_id;
  *xnew = kDead;
  if (lane == 0) {
    *xnew = compress_id(raw[b], tmap, c, status);
    slot = *xnew;
  } else if (lane < static_cast<uint32_t>(c.max_ngram) && !pad) {
    slot = check_hist(hist[static_cast<int64_t>(sl) * depth + (lane - 1)], c, status);
  }
  *pad_row = pad;
  return slot;
}

// Commit of decode entry b after every lane has consumed its window slot:
// (h0, h1, ...) <- (x', h0, ...).  Lane i holds g_i = x'_{t-i}, which is the
// new history entry i (most recent first).
__device__ __forceinline__ void step_commit(const HashConsts& c, int64_t b, const int32_t* __restrict__ slots,
                                            int32_t* hist, bool pad_row, int32_t xnew, int32_t slot) {
  const uint32_t lane = lane_id();
  const int depth = c.max_ngram - 1;
  if (!pad_row && lane < static_cast<uint32_t>(depth))
    hist[static_cast<int64_t>(slots[b]) * depth + lane] = (lane == 0) ? xnew : slot;
}

// Launches the history commit of a prefill chunk (hash.cu): the last
// max_ngram-1 compressed ids of each sequence, most recent first.
int launch_hist_commit(const HashConsts& c, const int32_t* raw, const int64_t* cu, int32_t n_seqs,
                       const int32_t* tmap, int32_t* hist, int32_t* status, cudaStream_t st);

}  // namespace hashdev
}  // namespace engram
