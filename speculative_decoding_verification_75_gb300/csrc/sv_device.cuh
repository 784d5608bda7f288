// sv_device.cuh -- device helpers for the verification kernels (sm_103a).
//
// Inline PTX for the Blackwell data-movement path (mbarrier, 1-D TMA bulk
// copies, programmatic dependent launch), bounded waits, element traits for
// fp32 / bf16 logits and warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "spec_verify.h"

namespace sv {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- PTX ----

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(tx)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A wait that cannot hang: gives up after ~2 s (or 2^30 polls), records
// SV_FAULT_TIMEOUT in the error word and returns false.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            uint32_t *err) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) break;
  }
  atomicOr(err, SV_FAULT_TIMEOUT);
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint32_t *err) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, err);
}

// L2 policy for streams read exactly once.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction count on
// the mbarrier.  src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const void *src,
                                            uint32_t bytes, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's completion
// (and memory flush), and allow the next grid to start its prologue.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2^x on the special-function unit (ftz: results below 2^-126 become 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ elements ----

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xffff0000u);
}

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kChunk = 4096;  // elements per 16 KiB chunk
  __device__ __forceinline__ static float load(const float *p, size_t i) {
    return __ldg(p + i);
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kChunk = 8192;
  __device__ __forceinline__ static float load(const __nv_bfloat16 *p, size_t i) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
};

// ----------------------------------------------------------- reductions ----

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Inclusive prefix sum over the lanes (fixed order: Hillis-Steele).
__device__ __forceinline__ float warp_inclusive_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Arrival counting for last-arriver merges: the add releases this thread's
// earlier writes and acquires everything released by earlier adders.
__device__ __forceinline__ uint32_t atomic_add_acq_rel(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Loads that bypass L1 (data written by other CTAs of the same grid), for
// any trivially copyable type made of 4-byte words.
template <typename T>
__device__ __forceinline__ T ld_cg(const T *p) {
  static_assert(sizeof(T) % 4 == 0, "word-sized types only");
  T out;
  if constexpr (sizeof(T) % 16 == 0 && alignof(T) >= 16) {
    const int4 *s = reinterpret_cast<const int4 *>(p);
    int4 *d = reinterpret_cast<int4 *>(&out);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(T) / 16); ++i) d[i] = __ldcg(s + i);
  } else if constexpr (sizeof(T) % 8 == 0 && alignof(T) >= 8) {
    const int2 *s = reinterpret_cast<const int2 *>(p);
    int2 *d = reinterpret_cast<int2 *>(&out);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(T) / 8); ++i) d[i] = __ldcg(s + i);
  } else {
    const int *s = reinterpret_cast<const int *>(p);
    int *d = reinterpret_cast<int *>(&out);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(T) / 4); ++i) d[i] = __ldcg(s + i);
  }
  return out;
}

}  // namespace sv
