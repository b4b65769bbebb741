// Host-resident table: gathering rows on the Grace side.
//
// Pages cited by title:
//   [P-V41] "DeepSeek-V4.1 模型结构（5）：记忆，Engram" §"196B 参数怎么存、怎么取"
//           (the rows to fetch depend only on token ids, so the table can live in
//           host memory and be fetched while earlier layers compute)
//   [P-O1]  "条件记忆：DeepSeek V4.1 Engram 如何用 O(1) 查表换掉一层计算" §4.1
//           (one gather serves device, pinned-host and ATS tables) and §五
//   [P-DETAIL] "DeepSeek Engram 详解：把静态知识从计算里拆出来" §8.2 (prefetch
//           overlapped with the earlier blocks' compute)
//
// On GB300 the table can stay in the Grace LPDDR and be read in two ways:
//   * directly by the gather kernel through NVLink-C2C (a pinned or ATS
//     pointer passed to engram_gather_dequant), or
//   * by host threads that copy the needed 264-byte rows into one contiguous
//     pinned staging buffer, which a single DMA then moves to HBM; the
//     dequantisation reads it with engram_dequant_rows.  This file is that
//     host gather; engram_host_gather_async orders it on a CUDA stream (after
//     the device-to-host copy of the row ids, before the host-to-device copy of
//     the staging buffer) so the whole fetch runs on the host cores and copy
//     engines, concurrently with kernels on other streams.
#include <cuda_runtime.h>
#include <omp.h>
#include <stdint.h>

#include <cstring>

#include "engram_internal.h"

namespace engram {
namespace {

struct HostGatherJob {
  const uint8_t* table;
  int64_t total_rows;
  const int32_t* row_ids;
  int64_t n_rows;
  uint8_t* staging;
  int n_threads;
  int64_t* bad_rows;  // may be null
};

// Copies row j.row_ids[i] to slot i of the staging buffer; returns 1 for an
// id outside the table (its slot is zeroed and dequantises to +0).
inline int64_t copy_row(const HostGatherJob& j, int64_t i) {
  const int64_t r = j.row_ids[i];
  uint8_t* dst = j.staging + i * ENGRAM_ROW_BYTES;
  if (r < 0 || r >= j.total_rows) {
    std::memset(dst, 0, ENGRAM_ROW_BYTES);
    return 1;
  }
  std::memcpy(dst, j.table + r * ENGRAM_ROW_BYTES, ENGRAM_ROW_BYTES);
  return 0;
}

// Rows are 264 bytes at random places in a table far larger than the host's
// caches, so a copy loop waits on memory latency; touching the rows a fixed
// distance ahead keeps several misses in flight per thread.
constexpr int64_t kPrefetchAhead = 12;

inline void prefetch_row(const HostGatherJob& j, int64_t i) {
  const int64_t r = j.row_ids[i];
  if (r < 0 || r >= j.total_rows) return;
  const uint8_t* p = j.table + r * ENGRAM_ROW_BYTES;
  for (int b = 0; b < ENGRAM_ROW_BYTES; b += 64) __builtin_prefetch(p + b, 0, 0);
  __builtin_prefetch(p + ENGRAM_ROW_BYTES - 1, 0, 0);
}

// Rows are handed out in chunks on demand: the calling thread and the other
// host work (a thread spinning on a CUDA event, say) share the cores with the
// team, and a fixed split would wait for whichever thread lost its core.
constexpr int64_t kChunkRows = 256;

int64_t run_host_gather(const HostGatherJob& j) {
  int64_t bad = 0;
  const int threads = j.n_threads > 0 ? j.n_threads : omp_get_max_threads();
  const int64_t n_chunks = (j.n_rows + kChunkRows - 1) / kChunkRows;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1) reduction(+ : bad)
  for (int64_t c = 0; c < n_chunks; ++c) {
    const int64_t lo = c * kChunkRows, hi = lo + kChunkRows < j.n_rows ? lo + kChunkRows : j.n_rows;
    for (int64_t i = lo; i < hi && i < lo + kPrefetchAhead; ++i) prefetch_row(j, i);
    for (int64_t i = lo; i < hi; ++i) {
      if (i + kPrefetchAhead < hi) prefetch_row(j, i + kPrefetchAhead);
      bad += copy_row(j, i);
    }
  }
  return bad;
}

void CUDART_CB host_gather_callback(void* user) {
  HostGatherJob* j = static_cast<HostGatherJob*>(user);
  int64_t bad = run_host_gather(*j);
  if (j->bad_rows) __atomic_store_n(j->bad_rows, bad, __ATOMIC_RELEASE);
  delete j;
}

int check_args(const uint8_t* table_h, int64_t total_rows, const int32_t* row_ids_h, int64_t n_rows,
               const uint8_t* staging_h) {
  if (n_rows < 0 || total_rows < 0) return fail(ENGRAM_E_INVALID, "negative size");
  if (n_rows > 0 && (!table_h || !row_ids_h || !staging_h)) return fail(ENGRAM_E_INVALID, "null host pointer");
  return ENGRAM_OK;
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" int engram_host_gather(const uint8_t* table_h, int64_t total_rows, const int32_t* row_ids_h,
                                  int64_t n_rows, uint8_t* staging_h, int32_t n_threads, int64_t* bad_rows) {
  int rc = check_args(table_h, total_rows, row_ids_h, n_rows, staging_h);
  if (rc) return rc;
  HostGatherJob j{table_h, total_rows, row_ids_h, n_rows, staging_h, n_threads, bad_rows};
  const int64_t bad = run_host_gather(j);
  if (bad_rows) *bad_rows = bad;
  return ENGRAM_OK;
}

extern "C" int engram_host_gather_async(const uint8_t* table_h, int64_t total_rows, const int32_t* row_ids_h,
                                        int64_t n_rows, uint8_t* staging_h, int32_t n_threads, int64_t* bad_rows,
                                        void* stream) {
  int rc = check_args(table_h, total_rows, row_ids_h, n_rows, staging_h);
  if (rc) return rc;
  if (n_rows == 0) return ENGRAM_OK;
  HostGatherJob* j = new HostGatherJob{table_h, total_rows, row_ids_h, n_rows, staging_h, n_threads, bad_rows};
  cudaError_t err = cudaLaunchHostFunc(as_stream(stream), host_gather_callback, j);
  if (err != cudaSuccess) {
    delete j;
    return fail(ENGRAM_E_CUDA, "cudaLaunchHostFunc: %s", cudaGetErrorString(err));
  }
  return ENGRAM_OK;
}
