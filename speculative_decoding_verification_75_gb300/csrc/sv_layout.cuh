// sv_layout.cuh -- workspace layout, vocabulary tiling and launch parameters.
//
// The caller-owned workspace holds everything kernel 0 and the CTAs of the
// persistent kernel hand to one another: per-request row offsets and softmax
// scales, arrival counters, the work counters of the persistent kernel's two
// queues, per-chunk partial statistics of the target softmax, the
// descriptors of the rows to re-sample and the per-chunk / per-segment
// residual sums that the inverse-CDF search walks.
#pragma once

#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>

#include "spec_verify.h"
#include "sv_device.cuh"

namespace sv {

// Every shared-memory stage holds one work item: a row-statistics chunk
// fills it with logits, a residual chunk with logits plus q (fp32).
#ifndef SV_STAGE_BYTES
#define SV_STAGE_BYTES 24576
#endif
constexpr int kStageBytes = SV_STAGE_BYTES;
constexpr int kSeg = 1024;  // elements per residual segment

template <typename T>
struct Tiling {
  static constexpr int kRowChunk = kStageBytes / static_cast<int>(sizeof(T));
  static constexpr int kResChunk =
      kStageBytes / (static_cast<int>(sizeof(T)) + 4) / kSeg * kSeg;
  static constexpr int kSegPerChunk = kResChunk / kSeg;
  static_assert(kRowChunk % 8 == 0 && kResChunk >= kSeg, "chunk shapes");
};
constexpr int kMinRowChunk = kStageBytes / 4;                // fp32 logits
constexpr int kMinResChunk = kStageBytes / 8 / kSeg * kSeg;  // fp32 logits + q

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kQFloor = 1e-10f;  // clamp of the acceptance divisor

struct __align__(128) Header {  // 512 bytes: four 128-byte lines
  uint32_t err;       // SV_BAD_* | SV_FAULT_* bits of this call
  uint32_t n_rows;    // active rows over all requests
  uint32_t n_valid;   // requests with rows (each is merged once)
  uint32_t a_next;    // next row-statistics item to hand out
  uint32_t pad0[28];  // the residual queue sits on its own 128-byte line
  uint32_t b_next;      // next residual item to hand out: chunk c of the
                        // descriptor in slot s is item s * C2 + c
  uint32_t b_reserved;  // descriptor slots reserved (read with b_next)
  uint32_t n_merged;    // requests merged so far
  uint32_t pad1[29];
  uint32_t jq_head;   // job tickets handed out
  uint32_t pad2[31];
  uint32_t all_merged;  // set by the last merge: b_reserved is final
  uint32_t pad3[31];    // (a line that is only read until then)
};

// jflag[j]: job j not (yet) due / due / never due.  Job b < B merges request
// b; job B + s searches the residual of descriptor slot s.
constexpr uint32_t kJobWait = 0u, kJobDue = 1u, kJobNone = 2u;

// State of descriptor slot s: reserved but not yet written / holds a row to
// re-sample / holds nothing (its request turned out invalid).
constexpr uint32_t kPending = 0u, kReadySample = 1u, kReadySkip = 2u;

struct __align__(8) Part {  // per (row, chunk) partial statistics
  float m;                  // chunk maximum logit
  float v;                  // sum exp2((l - m) * cs), or argmax bits
};

// Descriptor of one row to re-stream for the residual / bonus draw.
struct __align__(16) Desc {
  int b;        // request
  int k;        // first rejected position (g_b: bonus)
  int slot;     // padded row index of row k
  int tok;      // drafted token at k (one-hot q), or -1
  float m;      // row maximum logit
  float inv_s;  // 1 / normaliser
  float cs;     // log2(e) / T
  float u;      // sampling uniform
};
static_assert(sizeof(Desc) == 32, "eight 32-bit fields");

// A descriptor slot holds the eight fields of a Desc in eight 64-bit words,
// field i in the low half of word i and the slot's state in the high half.
// The merge writes the words with relaxed 64-bit stores (each single-copy
// atomic) and no fence; a reader takes the slot once every word carries the
// state: a word can only show the state together with its own field, so no
// release/acquire pair (a fence on each side, ~1-2 us under streaming load)
// stands between a merge and the residual work it publishes.
constexpr int kDescWords = 8;

__device__ __forceinline__ void desc_publish(uint64_t *w, const Desc &d, uint32_t state) {
  const uint32_t *f = reinterpret_cast<const uint32_t *>(&d);
#pragma unroll
  for (int i = 0; i < kDescWords; ++i)
    st_relaxed64(w + i, (static_cast<uint64_t>(state) << 32) | f[i]);
}


// One poll of a slot: all eight words in one round trip.  kReadySample only
// once every word carries it (d is then complete), kReadySkip as word 0
// shows it, else kPending.
__device__ __forceinline__ uint32_t desc_poll(const uint64_t *w, Desc &d) {
  uint32_t *f = reinterpret_cast<uint32_t *>(&d);
  uint64_t v[kDescWords];
#pragma unroll
  for (int i = 0; i < kDescWords; ++i) v[i] = ld_relaxed64(w + i);
  const uint32_t s0 = static_cast<uint32_t>(v[0] >> 32);
  if (s0 != kReadySample) return s0;
  bool all = true;
#pragma unroll
  for (int i = 0; i < kDescWords; ++i) {
    all = all && static_cast<uint32_t>(v[i] >> 32) == kReadySample;
    f[i] = static_cast<uint32_t>(v[i]);
  }
  return all ? kReadySample : kPending;
}

// Waits (bounded) until every word of a kReadySample slot has landed.
__device__ __forceinline__ bool desc_read(const uint64_t *w, Desc &d, uint32_t *err) {
  uint32_t *f = reinterpret_cast<uint32_t *>(&d);
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint64_t v[kDescWords];
#pragma unroll
    for (int i = 0; i < kDescWords; ++i) v[i] = ld_relaxed64(w + i);
    bool all = true;
#pragma unroll
    for (int i = 0; i < kDescWords; ++i) {
      all = all && static_cast<uint32_t>(v[i] >> 32) == kReadySample;
      f[i] = static_cast<uint32_t>(v[i]);
    }
    if (all) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, SV_FAULT_TIMEOUT);
      return false;
    }
  }
}


// Byte offsets of each region inside the workspace.
struct Layout {
  size_t hdr, row_start, cs, k1_cnt, k2_cnt, desc, jflag, part1, csum, ssum, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

inline int div_up(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Residual segment slots per row: whole chunks of whole segments.
template <typename T>
inline size_t seg_slots(int V) {
  return static_cast<size_t>(div_up(V, Tiling<T>::kResChunk)) * Tiling<T>::kSegPerChunk;
}

inline Layout make_layout(int B, int gmax, int V) {
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(gmax + 1);
  const size_t c1 = static_cast<size_t>(div_up(V, kMinRowChunk));
  const size_t c2 = static_cast<size_t>(div_up(V, kMinResChunk));
  const size_t sb = seg_slots<__nv_bfloat16>(V), sf = seg_slots<float>(V);
  const size_t nseg = sb > sf ? sb : sf;
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.hdr = take(sizeof(Header));
  L.row_start = take(sizeof(int) * (static_cast<size_t>(B) + 1));
  L.cs = take(sizeof(float) * B);
  L.k1_cnt = take(sizeof(uint32_t) * B);
  L.k2_cnt = take(sizeof(uint32_t) * B);
  L.desc = take(sizeof(uint64_t) * kDescWords * B);
  L.jflag = take(sizeof(uint32_t) * 2 * static_cast<size_t>(B));
  L.part1 = take(sizeof(Part) * rows * c1);
  L.csum = take(sizeof(float2) * B * c2);
  L.ssum = take(sizeof(float2) * B * nseg);
  L.total = o;
  return L;
}

// Everything a kernel needs, passed by value.
struct Params {
  const void *logits;
  const int32_t *ids;
  const float *q;
  const float *u_acc;
  const float *u_smp;
  const float *temp;
  const int32_t *lens;
  int B, gmax, V;
  int C1;    // row-statistics chunks per row
  int C2;    // residual chunks per row
  int nseg;  // residual segment slots per row (chunks * segments per chunk)
  int32_t *out_tokens;
  int32_t *out_nacc;
  sv_diag diag;
  Header *hdr;
  int *row_start;    // [B+1] first flat row of each request
  float *cs;         // [B] log2(e) / T (0: greedy)
  uint32_t *k1_cnt;  // [B] row-statistics chunks completed
  uint32_t *k2_cnt;  // [B] residual chunks completed
  uint64_t *desc;    // [B][kDescWords] rows to re-sample, in reservation (merge) order
  uint32_t *jflag;   // [2B] kJobWait / kJobDue / kJobNone per job
  Part *part1;
  float2 *csum;      // [slot][C2] residual and p sums per chunk
  float2 *ssum;      // [slot][nseg] residual and p sums per 1024-element segment
};

// Input checks shared by the kernels.
__device__ __forceinline__ bool valid_uniform(float u) { return u >= 0.f && u < 1.f; }

// 0 (greedy) or a normal, finite, positive binary32 value.
__device__ __forceinline__ bool valid_temperature(float t) {
  return t == 0.f || (t >= 1.17549435e-38f && t <= 3.40282347e38f);
}

// Rows of request b that are read (0 for an invalid draft length).
__device__ __forceinline__ int request_rows(const Params &p, int b) {
  if (!p.lens) return p.gmax + 1;
  const int g = __ldg(p.lens + b);
  return (g >= 0 && g <= p.gmax) ? g + 1 : 0;
}

}  // namespace sv
