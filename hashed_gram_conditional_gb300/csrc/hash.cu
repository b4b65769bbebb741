// Stages 1-3 of the Engram lookup: token map, suffix window with pad/DEAD,
// multiplicative-XOR mix and per-column prime modulo plus segment offset.
//
// Pages cited by title:
//   [P-V41]    "DeepSeek-V4.1 模型结构（5）：记忆，Engram"
//   [P-LMNT]   "Engram条件记忆：DeepSeek-V4.1-Flash中196B稀疏参数N-gram哈希查表的实现原理"
//   [P-O1]     "条件记忆：DeepSeek V4.1 Engram 如何用 O(1) 查表换掉一层计算"
//   [P-DS4]    "ds4.c 学习笔记" -- glossary entry "Engram"
//   [P-DETAIL] "DeepSeek Engram 详解：把静态知识从计算里拆出来"
//
// Work mapping: one warp per position.  Lanes 0..max_ngram-1 fetch the window
// slots, the slots are broadcast with shuffles, and lane j < n_cols computes
// column j, so the 24 row ids of a position leave as one 96-byte store.
#include <cuda_runtime.h>
#include <stdint.h>

#include "engram_internal.h"
#include "hash_device.cuh"

namespace engram {
using namespace hashdev;
namespace {

__global__ void __launch_bounds__(256) hash_prefill_kernel(
    HashConsts c, const int32_t* __restrict__ raw, int64_t n_tokens,
    const int64_t* __restrict__ cu, int32_t n_seqs, const int32_t* __restrict__ tmap,
    const int32_t* __restrict__ hist, int32_t* __restrict__ rows, uint8_t* __restrict__ mask,
    int32_t* status) {
  allow_dependent_launch();  // the history commit may load its inputs meanwhile
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
       t < n_tokens; t += warps) {
    const int32_t slot = prefill_slot(c, t, raw, cu, n_seqs, tmap, hist, status);
    hash_window(slot, c, rows + t * c.n_cols, mask + t, false);
  }
}

// Every Engram layer of the layout in one pass over the tokens: the window
// (token map, history, pad, DEAD cascade) does not depend on the layer, only
// the multipliers, primes and offsets do ([P-O1] §2.4: the indices depend
// only on the token ids, so all layers are hashed before the layer loop).
struct HashConstsAll {
  HashConsts l[ENGRAM_MAX_LAYERS];
  int32_t n_layers;
};

__global__ void __launch_bounds__(256) hash_all_layers_kernel(
    HashConstsAll ca, const int32_t* __restrict__ raw, int64_t n_tokens, const int64_t* __restrict__ cu,
    int32_t n_seqs, const int32_t* __restrict__ tmap, const int32_t* __restrict__ hist,
    int32_t* __restrict__ rows, uint8_t* __restrict__ mask, int32_t* status) {
  const HashConsts& c = ca.l[0];
  allow_dependent_launch();  // the history commit may load its inputs meanwhile
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; t < n_tokens;
       t += warps) {
    const int32_t slot = prefill_slot(c, t, raw, cu, n_seqs, tmap, hist, status);
    for (int li = 0; li < ca.n_layers; ++li)
      hash_window(slot, ca.l[li], rows + (static_cast<int64_t>(li) * n_tokens + t) * c.n_cols, mask + t, false);
  }
}

// History after a chunk: the last `depth` compressed ids of each sequence,
// most recent first, falling back to the previous history for short chunks.
// One thread per sequence reads all it needs before writing its own row.
// It is launched as a programmatic dependent of the kernel that hashed the
// chunk.  No kernel of the path writes the raw ids, the sequence bounds or the
// token map, so those loads run early; the old history is read, and the new
// one written, only once that kernel has finished (it reads the old history,
// and a decode-step gather before it would be writing it).
__global__ void hash_commit_kernel(HashConsts c, const int32_t* __restrict__ raw,
                                   const int64_t* __restrict__ cu, int32_t n_seqs,
                                   const int32_t* __restrict__ tmap, int32_t* hist,
                                   int32_t* status) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = s < n_seqs;
  const int depth = c.max_ngram - 1;
  const int64_t start = live ? cu[s] : 0, end = live ? cu[s + 1] : 0;
  const int64_t len = end - start;
  int32_t nh[ENGRAM_MAX_NGRAM - 1];
#pragma unroll
  for (int i = 0; i < ENGRAM_MAX_NGRAM - 1; ++i) {
    if (i >= depth) break;
    const int64_t pos = end - 1 - i;
    if (live && pos >= start) nh[i] = compress_id(raw[pos], tmap, c, nullptr);  // errors reported by the hash
  }
  wait_prior_grids();  // every position of the chunk has read the old history
  if (!live) return;
#pragma unroll
  for (int i = 0; i < ENGRAM_MAX_NGRAM - 1; ++i) {
    if (i >= depth) break;
    const int64_t pos = end - 1 - i;
    if (pos < start) nh[i] = hist[static_cast<int64_t>(s) * depth + (i - len)];
  }
#pragma unroll
  for (int i = 0; i < ENGRAM_MAX_NGRAM - 1; ++i) {
    if (i >= depth) break;
    hist[static_cast<int64_t>(s) * depth + i] = nh[i];
  }
}

// Decode step: warp per batch entry; the entry's history row is read by the
// first lanes, hashed, and rolled forward by lane 0 ([P-O1] §4.4: hash and
// history commit in one launch; padding entries commit nothing).
__global__ void __launch_bounds__(256) hash_step_kernel(
    HashConsts c, const int32_t* __restrict__ raw, const int32_t* __restrict__ slots, int32_t batch,
    const int32_t* __restrict__ tmap, int32_t* hist, int64_t n_slots, int32_t* __restrict__ rows,
    uint8_t* __restrict__ mask, int32_t* status) {
  const int b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (b >= batch) return;
  bool pad_row;
  int32_t xnew;
  const int32_t slot = step_slot(c, b, raw, slots, tmap, hist, n_slots, status, &pad_row, &xnew);
  // Every lane's history read has been consumed by the shuffles inside
  // hash_window before any lane writes the row below.
  hash_window(slot, c, rows + static_cast<int64_t>(b) * c.n_cols, mask + b, pad_row);
  __syncwarp();
  step_commit(c, b, slots, hist, pad_row, xnew, slot);
}

__global__ void selftest_mod_kernel(HashConsts c, const uint64_t* __restrict__ x, int64_t n,
                                    int64_t* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint64_t v = x[i];
  for (int j = 0; j < c.n_cols; ++j)
    out[i * c.n_cols + j] = static_cast<int64_t>(mod_prime(v, c.prime[j], c.recip[j])) + c.offset[j];
}

}  // namespace

int hashdev::launch_hist_commit(const HashConsts& c, const int32_t* raw, const int64_t* cu, int32_t n_seqs,
                                const int32_t* tmap, int32_t* hist, int32_t* status, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n_seqs + 127) / 128));
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, hash_commit_kernel, c, raw, cu, n_seqs, tmap, hist, status);
  if (err != cudaSuccess) return fail(ENGRAM_E_CUDA, "hash_commit_kernel launch: %s", cudaGetErrorString(err));
  return check_launch("hash_commit_kernel");
}

}  // namespace engram

using namespace engram;

extern "C" int engram_hash(const engram_layout* layout, int32_t layer, const int32_t* raw_ids_d,
                           int64_t n_tokens, const int64_t* cu_seqlens_d, int32_t n_seqs,
                           const int32_t* token_map_d, int64_t vocab_raw, int32_t* hist_d,
                           int32_t* row_ids_d, uint8_t* mask_d, int32_t* status_d, void* stream) {
  HashConsts c;
  int rc = make_consts(layout, layer, vocab_raw, &c);
  if (rc) return rc;
  if (n_tokens < 0 || n_seqs < 1) return fail(ENGRAM_E_INVALID, "n_tokens < 0 or n_seqs < 1");
  if (n_tokens == 0 && hist_d == nullptr) return ENGRAM_OK;
  if (!cu_seqlens_d || !token_map_d || (n_tokens > 0 && (!raw_ids_d || !row_ids_d || !mask_d)))
    return fail(ENGRAM_E_INVALID, "null device pointer");
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  cudaStream_t st = as_stream(stream);
  if (n_tokens > 0) {
    const int threads = 256;
    const int64_t want = (n_tokens + 7) / 8;
    const int blocks = static_cast<int>(want < int64_t(sms) * 16 ? want : int64_t(sms) * 16);
    hash_prefill_kernel<<<blocks, threads, 0, st>>>(c, raw_ids_d, n_tokens, cu_seqlens_d, n_seqs,
                                                    token_map_d, hist_d, row_ids_d, mask_d,
                                                    status_d);
    if ((rc = check_launch("hash_prefill_kernel"))) return rc;
  }
  if (hist_d != nullptr)
    return launch_hist_commit(c, raw_ids_d, cu_seqlens_d, n_seqs, token_map_d, hist_d, status_d, st);
  return ENGRAM_OK;
}

extern "C" int engram_hash_step(const engram_layout* layout, int32_t layer,
                                const int32_t* raw_ids_d, const int32_t* slots_d, int32_t batch,
                                const int32_t* token_map_d, int64_t vocab_raw, int32_t* hist_d,
                                int64_t n_slots, int32_t* row_ids_d, uint8_t* mask_d,
                                int32_t* status_d, void* stream) {
  HashConsts c;
  int rc = make_consts(layout, layer, vocab_raw, &c);
  if (rc) return rc;
  if (batch < 0 || n_slots < 0) return fail(ENGRAM_E_INVALID, "negative batch or n_slots");
  if (batch == 0) return ENGRAM_OK;
  if (!raw_ids_d || !slots_d || !token_map_d || !row_ids_d || !mask_d || (n_slots > 0 && !hist_d))
    return fail(ENGRAM_E_INVALID, "null device pointer");
  if ((rc = check_device(nullptr))) return rc;
  const int wpb = 8;
  hash_step_kernel<<<(batch + wpb - 1) / wpb, wpb * 32, 0, as_stream(stream)>>>(
      c, raw_ids_d, slots_d, batch, token_map_d, hist_d, n_slots, row_ids_d, mask_d, status_d);
  return check_launch("hash_step_kernel");
}

extern "C" int engram_selftest_mod(const engram_layout* layout, int32_t layer, const uint64_t* x_d,
                                   int64_t n, int64_t* out_d, void* stream) {
  HashConsts c;
  int rc = make_consts(layout, layer, 1, &c);
  if (rc) return rc;
  if (n < 0) return fail(ENGRAM_E_INVALID, "n < 0");
  if (n == 0) return ENGRAM_OK;
  if (!x_d || !out_d) return fail(ENGRAM_E_INVALID, "null device pointer");
  if ((rc = check_device(nullptr))) return rc;
  selftest_mod_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, as_stream(stream)>>>(c, x_d, n,
                                                                                            out_d);
  return check_launch("selftest_mod_kernel");
}

extern "C" int engram_hash_all_layers(const engram_layout* layout, const int32_t* raw_ids_d, int64_t n_tokens,
                                      const int64_t* cu_seqlens_d, int32_t n_seqs, const int32_t* token_map_d,
                                      int64_t vocab_raw, int32_t* hist_d, int32_t* row_ids_d, uint8_t* mask_d,
                                      int32_t* status_d, void* stream) {
  if (layout == nullptr) return fail(ENGRAM_E_INVALID, "null layout");
  HashConstsAll ca;
  ca.n_layers = layout->n_layers;
  for (int li = 0; li < layout->n_layers; ++li) {
    int rc = make_consts(layout, li, vocab_raw, &ca.l[li]);
    if (rc) return rc;
  }
  if (n_tokens < 0 || n_seqs < 1) return fail(ENGRAM_E_INVALID, "n_tokens < 0 or n_seqs < 1");
  if (n_tokens == 0 && hist_d == nullptr) return ENGRAM_OK;
  if (!cu_seqlens_d || !token_map_d || (n_tokens > 0 && (!raw_ids_d || !row_ids_d || !mask_d)))
    return fail(ENGRAM_E_INVALID, "null device pointer");
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  cudaStream_t st = as_stream(stream);
  if (n_tokens > 0) {
    const int64_t want = (n_tokens + 7) / 8;
    const int blocks = static_cast<int>(want < int64_t(sms) * 16 ? want : int64_t(sms) * 16);
    hash_all_layers_kernel<<<blocks, 256, 0, st>>>(ca, raw_ids_d, n_tokens, cu_seqlens_d, n_seqs, token_map_d,
                                                   hist_d, row_ids_d, mask_d, status_d);
    if ((rc = check_launch("hash_all_layers_kernel"))) return rc;
  }
  if (hist_d != nullptr)
    return launch_hist_commit(ca.l[0], raw_ids_d, cu_seqlens_d, n_seqs, token_map_d, hist_d, status_d, st);
  return ENGRAM_OK;
}
