// Device-side helpers shared by the library's kernels: bf16 widening / rounding, the
// per-element Adam update, and thin PTX wrappers (mbarrier, bulk copies, timer). Streaming
// global accesses use the __ldcs / __stcs intrinsics (each byte is touched once per step).
//
// Every arithmetic step of the update uses an explicit round-to-nearest intrinsic
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn): the compiler never contracts these into
// fused multiply-adds, so each line rounds exactly once in IEEE fp32, and the library is
// additionally built with -fmad=false. No fast-math, no flush-to-zero.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace zgb {

// ------------------------------------------------------------------------------------
// device error word: first error wins; read and cleared by zero_device_status()
// ------------------------------------------------------------------------------------
// Codes: (kernel id << 8) | wait id. A bounded wait that gives up records its code,
// raises the CTA's abort flag and makes every role of that CTA leave its loop.
#define ZGB_DECLARE_ERROR_WORD() static __device__ unsigned int g_zgb_dev_error = 0u

// Timeout for any spin-wait on an mbarrier (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------------
// bf16 <-> fp32
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// round-to-nearest-even pair: first argument in the low half (lower address)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

// ------------------------------------------------------------------------------------
// the update of one element
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void adam_elem(float g, float& w, float& m, float& v, const AdamScalars& s) {
  const float m1 = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, g));
  const float v1 = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
  const float mh = __fdiv_rn(m1, s.bc1);
  const float vh = __fdiv_rn(v1, s.bc2);
  const float den = __fadd_rn(__fsqrt_rn(vh), s.eps);
  float x = w;
  if (s.wd_on) x = __fsub_rn(x, __fmul_rn(s.lr_wd, x));
  x = __fsub_rn(x, __fmul_rn(s.lr, __fdiv_rn(mh, den)));
  w = x;
  m = m1;
  v = v1;
}

// ------------------------------------------------------------------------------------
// shared memory, mbarrier and bulk-copy wrappers
// ------------------------------------------------------------------------------------
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
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete. Gives up after
// kWaitTimeoutNs or as soon as another thread of the CTA raised *abort; on a timeout it
// records `code` in the error word and raises *abort. Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  unsigned int* err_word, unsigned int code,
                                                  unsigned long long timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > timeout_ns) {
      atomicCAS(err_word, 0u, code);
      *abort = 1;
      return false;
    }
  }
}

// ---- thread-block clusters ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// every thread of every CTA of the cluster (no warp-convergence requirement)
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// arrive on an mbarrier given by its shared::cluster address (possibly in another CTA)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// mbar_try_wait with cluster-scope acquire: pairs with arrivals from other CTAs
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait_bounded with cluster-scope acquire
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                          unsigned int* err_word, unsigned int code) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > kWaitTimeoutNs) {
      atomicCAS(err_word, 0u, code);
      *abort = 1;
      return false;
    }
  }
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst_smem),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

}  // namespace zgb
