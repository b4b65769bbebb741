// Internal helpers of libengram: error reporting, device checks and the
// inline-PTX primitives (mbarrier, bulk copies, TMA, tcgen05) the kernels use.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/engram.h"

namespace engram {

// ---------------------------------------------------------------- host side

void set_error(const char* fmt, ...);
int fail(int code, const char* fmt, ...);
// Checks that the current device is an sm_103 GPU; fills the SM count.
int check_device(int* sm_count);
int check_launch(const char* what);
// The engram_kernel_options in force (engram_set_kernel_options).
engram_kernel_options kernel_options();

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Word of row (or column) i within a k-block row of a block-FP8 scale array:
// the words of each 128 consecutive rows are stored so that the 16 bytes at
// word 4 r hold rows r, r + 32, r + 64 and r + 96 -- the 32-row x 128-bit
// image that tcgen05.cp.32x128b.warpx4 spreads over the four TMEM lane
// quarters, in the layout the block-scaled MMA reads.
#ifdef __CUDACC__
__host__ __device__
#endif
inline int64_t sf_word_index(int64_t i) {
  return (i & ~int64_t(127)) | ((i & 31) << 2) | ((i >> 5) & 3);
}

// ------------------------------------------------------------- device side
#ifdef __CUDACC__

// Cycle budget of any on-chip wait.  Every kernel finishes in milliseconds;
// a wait that lasts ~2^31 cycles (about a second) means a broken invariant,
// and the kernel then records ENGRAM_ST_TIMEOUT and unwinds instead of hanging.
constexpr long long kWaitBudgetCycles = 1LL << 31;

// Programmatic dependent launch: a kernel launched right after this one with
// programmatic stream serialization may be scheduled once every CTA of this
// grid has issued this (its griddepcontrol.wait still waits for the whole
// grid to finish and its writes to be visible).
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits for the grids this one depends on programmatically (a no-op when the
// launch had no such dependency).
__device__ __forceinline__ void wait_prior_grids() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One test of the phase; a thread whose phase is not complete yet may be
// suspended (woken when the phase completes, at most kSuspendHintNs later)
// rather than spin, so waiting warps leave the issue slots of their SM
// sub-partition to the warps that work.
constexpr uint32_t kSuspendHintNs = 1000000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Pairs of fp32 values in one 64-bit register pair, for the packed
// two-lane fp32 instructions of sm_100+ (add/mul/fma .rn.f32x2): each lane
// is the IEEE round-to-nearest result of the scalar operation, so the packed
// code computes exactly what the scalar code does, in half the instructions.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Waits for the phase with the given parity to complete.  Returns false if
// the cycle budget ran out or *abort became nonzero (another role gave up).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (clock64() - t0 > kWaitBudgetCycles) return false;
  }
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled TMA load, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// SplitMix64 output number n+1 of a stream starting at `seed` (Steele, Lea &
// Flood 2014): finaliser applied to seed + (n+1) * golden gamma.  Used only by
// the synthetic-table generators (test and benchmark inputs).
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t n) {
  uint64_t z = seed + (n + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

#endif  // __CUDACC__

}  // namespace engram
