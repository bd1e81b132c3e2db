// Device-side helpers shared by the kvq kernels (sm_103a): error reporting,
// bounded mbarrier waits, 1-D bulk (TMA engine) copies, e4m3 conversions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq.h"

namespace kvq {

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------

__device__ __forceinline__ void report(uint32_t *err_word, uint32_t bit) {
  if (err_word) atomicOr(err_word, bit);
}

// ---------------------------------------------------------------------------
// shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------

// Programmatic dependent launch.  A kernel launched as a dependent (see
// launch_dependent) may become resident before the work ahead of it on the
// stream has finished; grid_dependency_wait() returns once that work has
// completed and its memory is visible, so it precedes every global-memory
// access of such a kernel.  allow_dependents() lets the next dependent
// launch be scheduled; it orders nothing by itself.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// A wait that gives up: about 2^31 SM cycles (~1 s at 2 GHz) or 2^24 polls,
// whichever comes first.  Returns false when it gave up.
constexpr long long kWaitCycles = 1LL << 31;
constexpr uint32_t kWaitPolls = 1u << 24;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitCycles) break;
  }
  return false;
}

// The drain of a CTA whose wait gave up: waits (bounded) for the copies of
// the ring stages before stage g that can still be in flight (the last ns)
// and for the last two of a double buffer of nq copies.  Out of line: the
// code never runs in a healthy call, and inlined it changed the split
// kernel's steady loop enough to cost ~0.6% at 64 requests.
static __device__ __noinline__ void drain_copies(uint64_t *full, uint32_t ns, uint32_t g,
                                                 uint64_t *qfull, uint32_t nq) {
  for (uint32_t k = g > ns ? g - ns : 0; k < g; ++k) mbar_wait(&full[k % ns], (k / ns) & 1);
  for (uint32_t k = nq > 2 ? nq - 2 : 0; k < nq; ++k) mbar_wait(&qfull[k & 1], (k >> 1) & 1);
}

// ---------------------------------------------------------------------------
// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Same, with an L2 eviction policy (streamed data that is read once).
__device__ __forceinline__ void bulk_g2s_hint(void *dst_smem, const void *src_gmem,
                                              uint32_t bytes, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// ---------------------------------------------------------------------------
// conversions
// ---------------------------------------------------------------------------

// two e4m3 codes (low byte = element 0) -> two fp16 (exact: e4m3 is a subset)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// four e4m3 codes in a 32-bit word -> four floats (exact)
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float *out) {
  const uint32_t lo = e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xFFFFu));
  const uint32_t hi = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
  const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
  out[0] = a.x;
  out[1] = a.y;
  out[2] = b.x;
  out[3] = b.y;
}

// two bf16 in a 32-bit word (low half = element 0) -> two floats (exact)
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float *out) {
  out[0] = __uint_as_float(w << 16);
  out[1] = __uint_as_float(w & 0xFFFF0000u);
}

// two floats -> two e4m3 codes, round to nearest even, saturating to +-448
// (low byte = `lo`)
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace kvq
