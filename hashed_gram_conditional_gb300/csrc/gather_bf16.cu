// Stage 4 for tables whose rows are plain bf16 vectors of any width that is a
// multiple of 8 elements -- the generic-shape row format.  The Engram paper's
// 27B configuration reads 16 rows of 80 elements per position (two n-gram
// orders x 8 heads, a 1280-wide concatenation) into a hidden size of 2560
// ([P-DETAIL] "DeepSeek Engram 详解" §5, after its worked example, quoting
// the paper's Table 5); the same page sizes such a table in bf16, 2 bytes per
// element (§8.4).  The DeepSeek-V4.1 table is E4M3 + E8M0 (gather.cu).
//
// A row is copied as it is: e[t][j*row_dim + c] = table[row_ids[t][j]][c].
// One warp per position; lane j < n_cols holds column j's row id, and the
// row's 16-byte pieces are spread over the lanes, all loads of a position
// issued before its stores.
#include <cuda_runtime.h>
#include <stdint.h>

#include "engram_internal.h"
#include "hash_device.cuh"

namespace engram {
namespace {

constexpr int kWarpsB = 8;   // warps per block
constexpr int kUnrollB = 5;  // 16-byte pieces in flight per lane per round: one round for 16 rows of 80

template <bool kHash>
__global__ void __launch_bounds__(kWarpsB * 32) gather_rows_bf16_kernel(
    const uint16_t* __restrict__ table, int64_t total_rows, int32_t row_dim, const int32_t* __restrict__ row_ids,
    int64_t n_tokens, int32_t n_cols, uint16_t* __restrict__ e, int32_t* status, hashdev::HashConsts c,
    const int32_t* __restrict__ raw, const int64_t* __restrict__ cu, int32_t n_seqs,
    const int32_t* __restrict__ tmap, const int32_t* __restrict__ hist, int32_t* rows_out, uint8_t* mask) {
  // Launched as a programmatic dependent: nothing is read before the
  // previous kernel has finished, and a following history commit may start
  // (and load its inputs) only after that, never ahead of this kernel's own
  // predecessor.
  wait_prior_grids();
  allow_dependent_launch();
  const uint32_t lane = lane_id();
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int per_row = row_dim / 8;  // 16-byte pieces per row
  const int pieces = n_cols * per_row;
  for (int64_t t = gw; t < n_tokens; t += nw) {
    int32_t r = -1;
    if (kHash) {
      const int32_t slot = hashdev::prefill_slot(c, t, raw, cu, n_seqs, tmap, hist, status);
      const bool dead = hashdev::window_rows(slot, c, &r);
      if (rows_out != nullptr && lane < static_cast<uint32_t>(n_cols)) rows_out[t * n_cols + lane] = r;
      if (lane == 0) mask[t] = dead ? 1 : 0;
    } else if (lane < static_cast<uint32_t>(n_cols)) {
      r = __ldg(row_ids + t * n_cols + lane);
    }
    const bool valid = lane < static_cast<uint32_t>(n_cols) && r >= 0 && static_cast<int64_t>(r) < total_rows;
    if (lane < static_cast<uint32_t>(n_cols) && !valid && status != nullptr)
      atomicOr(status, static_cast<int>(ENGRAM_ST_BAD_ROW));
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    uint4* out = reinterpret_cast<uint4*>(e + t * static_cast<int64_t>(pieces) * 8);
    for (int p0 = 0; p0 < pieces; p0 += 32 * kUnrollB) {
      uint4 v[kUnrollB];
#pragma unroll
      for (int u = 0; u < kUnrollB; ++u) {
        const int p = p0 + u * 32 + static_cast<int>(lane);
        const int j = p / per_row;
        const int32_t rr = __shfl_sync(0xffffffffu, r, j & 31);
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (p < pieces && ((vmask >> (j & 31)) & 1u))
          v[u] = __ldg(reinterpret_cast<const uint4*>(table + static_cast<int64_t>(rr) * row_dim) + (p - j * per_row));
      }
#pragma unroll
      for (int u = 0; u < kUnrollB; ++u) {
        const int p = p0 + u * 32 + static_cast<int>(lane);
        if (p < pieces) out[p] = v[u];
      }
    }
  }
}

// Synthetic bf16 rows: element c of row r is 16-bit piece (c mod 4) of
// SplitMix64 output number r*(row_dim/4) + c/4 + 1 of the stream at `seed`,
// with its 8 exponent bits replaced by 120 + (those bits mod 11) (finite
// values of magnitude in [2^-7, 2^4)).
__global__ void fill_rows_bf16_kernel(uint64_t* __restrict__ words, int64_t n_words, uint64_t seed) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint64_t z = splitmix64_at(seed, static_cast<uint64_t>(i));
    uint64_t o = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t b = static_cast<uint32_t>(z >> (16 * k)) & 0xffffu;
      const uint32_t ex = 120u + ((b >> 7) & 0xffu) % 11u;
      o |= static_cast<uint64_t>((b & 0x807fu) | (ex << 7)) << (16 * k);
    }
    words[i] = o;
  }
}

int check_rows_bf16(int64_t total_rows, int32_t row_dim, int32_t n_cols) {
  if (total_rows < 0) return fail(ENGRAM_E_INVALID, "negative size");
  if (row_dim < 8 || row_dim % 8 != 0 || row_dim > 4096)
    return fail(ENGRAM_E_SHAPE, "row_dim %d must be a multiple of 8 in [8, 4096]", row_dim);
  if (n_cols < 1 || n_cols > ENGRAM_MAX_COLS) return fail(ENGRAM_E_SHAPE, "n_cols %d", n_cols);
  return ENGRAM_OK;
}

int launch_rows_bf16(bool hash, const uint16_t* table_d, int64_t total_rows, int32_t row_dim,
                     const int32_t* row_ids_d, int64_t n_tokens, int32_t n_cols, uint16_t* e_d, int32_t* status_d,
                     const hashdev::HashConsts& c, const int32_t* raw, const int64_t* cu, int32_t n_seqs,
                     const int32_t* tmap, const int32_t* hist, int32_t* rows_out, uint8_t* mask, cudaStream_t st) {
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  const int64_t want = (n_tokens + kWarpsB - 1) / kWarpsB;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 64 warps per SM
  const int blocks = static_cast<int>(want < cap ? want : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kWarpsB * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the launch overlaps the previous kernel's tail
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaError_t err;
  if (hash)
    err = cudaLaunchKernelEx(&cfg, gather_rows_bf16_kernel<true>, table_d, total_rows, row_dim,
                             static_cast<const int32_t*>(nullptr), n_tokens, n_cols, e_d, status_d, c, raw, cu,
                             n_seqs, tmap, hist, rows_out, mask);
  else
    err = cudaLaunchKernelEx(&cfg, gather_rows_bf16_kernel<false>, table_d, total_rows, row_dim, row_ids_d, n_tokens,
                             n_cols, e_d, status_d, c, static_cast<const int32_t*>(nullptr),
                             static_cast<const int64_t*>(nullptr), 0, static_cast<const int32_t*>(nullptr),
                             static_cast<const int32_t*>(nullptr), static_cast<int32_t*>(nullptr),
                             static_cast<uint8_t*>(nullptr));
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "gather_rows_bf16_kernel launch: %s", cudaGetErrorString(err));
  return check_launch("gather_rows_bf16_kernel");
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" int engram_gather_rows_bf16(const uint16_t* table_d, int64_t total_rows, int32_t row_dim,
                                       const int32_t* row_ids_d, int64_t n_tokens, int32_t n_cols, uint16_t* e_d,
                                       int32_t* status_d, void* stream) {
  int rc = check_rows_bf16(total_rows, row_dim, n_cols);
  if (rc) return rc;
  if (n_tokens < 0) return fail(ENGRAM_E_INVALID, "n_tokens < 0");
  if (n_tokens == 0) return ENGRAM_OK;
  if (!table_d || !row_ids_d || !e_d) return fail(ENGRAM_E_INVALID, "null device pointer");
  if (!aligned(table_d, 16) || !aligned(e_d, 16)) return fail(ENGRAM_E_ALIGN, "table and e must be 16-byte aligned");
  hashdev::HashConsts c{};
  return launch_rows_bf16(false, table_d, total_rows, row_dim, row_ids_d, n_tokens, n_cols, e_d, status_d, c, nullptr,
                          nullptr, 0, nullptr, nullptr, nullptr, nullptr, as_stream(stream));
}

extern "C" int engram_hash_gather_rows_bf16(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                                            int64_t n_tokens, const int64_t* cu_seqlens_d, int32_t n_seqs,
                                            const int32_t* token_map_d, int64_t vocab_raw, int32_t* hist_d,
                                            const uint16_t* table_d, int32_t row_dim, uint16_t* e_d,
                                            uint8_t* mask_d, int32_t* row_ids_d, int32_t* status_d, void* stream) {
  hashdev::HashConsts c;
  int rc = hashdev::make_consts(layout, layer, vocab_raw, &c);
  if (rc) return rc;
  const int64_t total_rows = layout->total_rows[layer];
  if ((rc = check_rows_bf16(total_rows, row_dim, c.n_cols))) return rc;
  if (n_tokens < 0 || n_seqs < 1) return fail(ENGRAM_E_INVALID, "n_tokens < 0 or n_seqs < 1");
  if (n_tokens == 0 && hist_d == nullptr) return ENGRAM_OK;
  if (!cu_seqlens_d || !token_map_d || (n_tokens > 0 && (!raw_ids_d || !table_d || !e_d || !mask_d)))
    return fail(ENGRAM_E_INVALID, "null device pointer");
  if (n_tokens > 0 && (!aligned(table_d, 16) || !aligned(e_d, 16)))
    return fail(ENGRAM_E_ALIGN, "table and e must be 16-byte aligned");
  cudaStream_t st = as_stream(stream);
  if (n_tokens > 0 &&
      (rc = launch_rows_bf16(true, table_d, total_rows, row_dim, nullptr, n_tokens, c.n_cols, e_d, status_d, c,
                             raw_ids_d, cu_seqlens_d, n_seqs, token_map_d, hist_d, row_ids_d, mask_d, st)))
    return rc;
  // the history advances after every position has read the old one
  if (hist_d != nullptr)
    return hashdev::launch_hist_commit(c, raw_ids_d, cu_seqlens_d, n_seqs, token_map_d, hist_d, status_d, st);
  return ENGRAM_OK;
}

extern "C" int engram_fill_synthetic_rows_bf16(uint16_t* table_d, int64_t n_rows, int32_t row_dim, uint64_t seed,
                                               void* stream) {
  if (n_rows < 0) return fail(ENGRAM_E_INVALID, "n_rows < 0");
  if (row_dim < 4 || row_dim % 4 != 0) return fail(ENGRAM_E_SHAPE, "row_dim %d must be a multiple of 4", row_dim);
  if (n_rows == 0) return ENGRAM_OK;
  if (!table_d) return fail(ENGRAM_E_INVALID, "null table");
  if (!aligned(table_d, 8)) return fail(ENGRAM_E_ALIGN, "table must be 8-byte aligned");
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  const int64_t n_words = n_rows * (row_dim / 4);
  fill_rows_bf16_kernel<<<sms * 8, 256, 0, as_stream(stream)>>>(reinterpret_cast<uint64_t*>(table_d), n_words, seed);
  return check_launch("fill_rows_bf16_kernel");
}
