// mbarrier and bulk-copy primitives (inline PTX) shared by the kernels that
// stage logits in shared memory with cp.async.bulk: the TMA-pipelined verify
// scan (scan_tma.cu) and the cluster-per-row verify (cluster_select.cu).
// Every wait is bounded: a wait that runs out returns false, and a CTA never
// exits while a copy it issued may still be in flight (the drain).
#pragma once
#include <stdint.h>

namespace graft {
namespace bulk {

constexpr uint32_t SPIN = 1u << 22;     // try_wait polls before a wait gives up (unless the launch sets a limit)
constexpr uint32_t DRAIN = 1u << 20;    // back-off rounds (1 us each) the drain waits for a copy in flight

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// non-blocking check of the phase (try_wait may block for a hardware-defined
// interval; this does not, so a limit of n polls is n checks)
__device__ __forceinline__ bool mbar_test_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// whole warp, at most `polls` non-blocking checks, warp-uniform result
__device__ __forceinline__ bool mbar_poll_warp(unsigned long long* bar, uint32_t parity, uint32_t polls) {
  bool ok = false;
  for (uint32_t it = 0; it < polls; ++it) {
    ok = mbar_test_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
  }
  return __all_sync(0xffffffffu, ok);
}
// one thread, at most `polls` polls
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity, uint32_t polls) {
  for (uint32_t it = 0; it < polls; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// whole warp, at most `polls` polls, warp-uniform result
__device__ __forceinline__ bool mbar_wait_warp(unsigned long long* bar, uint32_t parity, uint32_t polls) {
  bool ok = false;
  for (uint32_t it = 0; it < polls; ++it) {
    ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
  }
  return __all_sync(0xffffffffu, ok);
}
// the drain: one thread waits for a copy it issued to land, backing off 1 us
// between polls, for about a second at most
__device__ __forceinline__ bool mbar_wait_drain(unsigned long long* bar, uint32_t parity) {
  for (uint32_t it = 0; it < DRAIN; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(1000);
  }
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

}  // namespace bulk
}  // namespace graft
