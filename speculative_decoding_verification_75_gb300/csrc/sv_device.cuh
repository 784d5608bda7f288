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

// Non-blocking test of a phase (try_wait may suspend the thread for a while;
// test_wait returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; "
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

// try_wait that lets the thread sleep in hardware until the phase completes
// (or about hint_ns pass), so waiting warps leave the issue slots and the
// memory pipeline to the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint32_t *err,
                                            uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = global_timer_ns();
  const uint32_t hint = limit_ns < 100000u ? static_cast<uint32_t>(limit_ns) : 100000u;
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait_sleep(bar, parity, hint)) return true;
    if (global_timer_ns() - t0 > limit_ns) break;
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

// Whole-warp wait on an mbarrier phase; false (for every lane) on timeout.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint32_t *err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err));
}

// ------------------------------------------------------- smem queues ----
// Single-producer single-consumer queue in shared memory: N entries of type
// E, each slot guarded by a "full" and an "empty" mbarrier (count 1).  One
// carries claimed work from a CTA's claimer lane to its producer lane, one
// carries completed runs from the producer lane to the service warp (so that
// merges and searches, several dependent memory round trips, never stall the
// streaming pipeline).
constexpr int kSvcSlots = 32;

template <typename E, int N = kSvcSlots>
struct SvcQueue {
  static constexpr int kSlots = N;
  E slot[N];
  uint64_t full[N];
  uint64_t empty[N];
};

template <typename Q>
__device__ __forceinline__ void svc_init(Q *q) {
  for (int i = 0; i < Q::kSlots; ++i) {
    mbar_init(smem_addr(&q->full[i]), 1);
    mbar_init(smem_addr(&q->empty[i]), 1);
  }
}

// Producer side (one thread), entry number k.  False on timeout.
template <typename Q, typename E>
__device__ __forceinline__ bool svc_push(Q *q, uint32_t k, const E &e, uint32_t *err) {
  constexpr uint32_t N = Q::kSlots;
  const int i = static_cast<int>(k % N);
  if (k >= N && !mbar_wait(smem_addr(&q->empty[i]), ((k / N) & 1u) ^ 1u, err)) return false;
  q->slot[i] = e;
  mbar_arrive(smem_addr(&q->full[i]));  // release: the entry and all the pusher observed
  return true;
}

// Programmatic dependent launch: wait for the preceding grid's completion
// (and memory flush), and allow the next grid to start its prologue.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block clusters: this CTA's rank, the cluster's size, a barrier of
// every thread of the cluster (release / acquire: shared-memory writes
// before it are visible to peers after it), and a load from a peer CTA's
// shared memory (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split form: arrive early (nothing to publish), wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_peer_f2(void *local, uint32_t rank, float2 v) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(ra), "f"(v.x), "f"(v.y) : "memory");
}
__device__ __forceinline__ float2 ld_peer_f2(const void *local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(ra) : "memory");
  return v;
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
  __device__ __forceinline__ static float load(const float *p, size_t i) {
    return __ldg(p + i);
  }
  // From shared memory (a plain load: the read-only path is global only).
  __device__ __forceinline__ static float load_shared(const float *p, int i) { return p[i]; }
};

template <>
struct Elem<__nv_bfloat16> {
  __device__ __forceinline__ static float load(const __nv_bfloat16 *p, size_t i) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  __device__ __forceinline__ static float load_shared(const __nv_bfloat16 *p, int i) {
    const unsigned short h = reinterpret_cast<const unsigned short *>(p)[i];
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

__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(uint32_t *p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add_release(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's earlier loads (that observed other threads' writes)
// before its later accesses, at device scope.
__device__ __forceinline__ void fence_acq_rel() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed64(uint64_t *p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed64(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release64(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire64(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Two adjacent 32-bit counters read in one access (8-byte aligned).
__device__ __forceinline__ uint2 ld_relaxed2(const uint32_t *p) {
  uint2 v;
  asm volatile("ld.relaxed.gpu.global.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p)
               : "memory");
  return v;
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
