// Device helpers shared by the TurboQuant kernels: inline-PTX wrappers for
// mbarriers, bulk (TMA) copies and cp.async, plus small math helpers.
// Every wait on the device is bounded: it polls at most `limit` times, then
// records kErrTimeout in the caller's error word and reports failure.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_internal.h"

namespace tq {

constexpr uint32_t kDefaultWaitLimit = 1u << 26;   // ~ seconds of polling

// ---- bounds-checked build ------------------------------------------------------
// Compiled with TQ_DEBUG_BOUNDS, every index a kernel computes into shared or
// global memory is checked against the extent of the buffer it addresses: an
// index outside it sets kErrBounds in the kernel's error word, and the access
// goes to the buffer's first element instead (a copy is dropped and its bytes
// are retired from its barrier), so nothing outside the buffer is touched and
// no wait is left hanging.  The normal build compiles the checks away.
#ifdef TQ_DEBUG_BOUNDS
constexpr bool kBoundsChecks = true;
#else
constexpr bool kBoundsChecks = false;
#endif

// p, or base when [p, p + sizeof(T)) leaves [base, base + bytes)
template <class T>
__device__ __forceinline__ T* bchk(T* p, const void* base, size_t bytes, unsigned* err) {
  if constexpr (kBoundsChecks) {
    const uintptr_t q = (uintptr_t)p, b0 = (uintptr_t)base;
    if (q < b0 || q + sizeof(T) > b0 + bytes) {
      atomicOr(err, kErrBounds);
      return (T*)base;
    }
  }
  return p;
}
// whether [p, p + n) lies inside [base, base + bytes) (always, in the normal build)
__device__ __forceinline__ bool bchk_range(const void* p, size_t n, const void* base,
                                           size_t bytes, unsigned* err) {
  if constexpr (kBoundsChecks) {
    const uintptr_t q = (uintptr_t)p, b0 = (uintptr_t)base;
    if (q < b0 || q + n > b0 + bytes) {
      atomicOr(err, kErrBounds);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- mbarrier ------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Retire `bytes` of a barrier's expected transaction count without a copy
// (the fault-injection hook's extra bytes, so that the drain after a timeout
// can see the real copies land).
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Bounded wait; returns false (and flags the error word) when it gives up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit,
                                          unsigned* err) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  atomicOr(err, kErrTimeout);
  return false;
}

// ---- bulk copy global -> shared (TMA, non-tensor form) ---------------------------
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- cp.async (per-thread asynchronous copies) ------------------------------------
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- shared loads -------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  uint32_t lsb = (u >> 16) & 1u;
  u = u + 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// In-register unnormalised Walsh-Hadamard transform of N values (Sylvester order).
template <int N>
__device__ __forceinline__ void fwht_regs(float (&x)[N]) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & h) == 0) {
        float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
}

// Code of coordinate I in a dense LSB-first stream held in 32-bit words.
template <int BITS, int I, int NW>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[NW]) {
  constexpr int p = I * BITS;
  constexpr int wi = p >> 5;
  constexpr int sh = p & 31;
  constexpr uint32_t mask = (1u << BITS) - 1u;
  if constexpr (sh + BITS <= 32) {
    return (w[wi] >> sh) & mask;
  } else {
    return ((w[wi] >> sh) | (w[wi + 1] << (32 - sh))) & mask;
  }
}

}  // namespace tq
