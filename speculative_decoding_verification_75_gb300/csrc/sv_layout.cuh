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
// 27 KiB: eight stages fill the shared memory the tables leave (24 KiB
// stages measured 64.0 vs 63.0 us for 128 requests of 6 bf16 rows of
// 151936 logits, 114.4 vs 107.8 us for 256 ragged requests).
#ifndef SV_STAGE_BYTES
#define SV_STAGE_BYTES 27648
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

// Work counters of one call.  Consecutive calls on a workspace alternate
// between two sets: a call runs on set (epoch & 1) while its CTA 0 clears
// set (epoch + 1) & 1 for the next call, so no call has to reset state that
// its own CTAs are about to use.
struct __align__(128) Counters {  // 512 bytes: four 128-byte lines
  uint32_t a_next;      // row-statistics items handed out after the static first blocks
  uint32_t pad0[31];
  uint32_t b_next;      // next residual item to hand out: chunk c of the
                        // descriptor in slot s is item s * C2 + c
  uint32_t b_reserved;  // descriptor slots reserved (read with b_next)
  uint32_t n_merged;    // requests finished (merged, or rejected for their length)
  uint32_t pad1[29];
  uint32_t jq_head;     // job tickets handed out
  uint32_t exited;      // CTAs that have finished
  uint32_t pad2[30];
  uint32_t all_merged;  // set by the last merge: b_reserved is final
  uint32_t pad3[31];    // (a line that is only read until then)
};

struct __align__(128) Header {
  uint32_t epoch;     // calls completed on this workspace (advanced by the last CTA out)
  uint32_t err[2];    // SV_BAD_* | SV_FAULT_* bits of the call with that epoch parity
  uint32_t pad0;
  uint64_t ready[2];  // certificate that counter set s is clear for the call it serves
  uint64_t pad1[13];
  Counters set[2];
};

static_assert(offsetof(Header, epoch) == 0 && offsetof(Header, err) == 4,
              "sv_last_error reads the epoch and both error words as three words");
static_assert(offsetof(Header, ready) % 8 == 0 && offsetof(Header, set) % 128 == 0 &&
                  offsetof(Counters, b_reserved) == offsetof(Counters, b_next) + 4,
              "header alignment");

// Certificate of counter set (e & 1) for the call with epoch e on a workspace
// laid out for (B, gmax, V): any other value in ready[] -- a fresh or
// foreign workspace, another layout, a call that faulted -- makes the call
// clear the set itself before using it.
__host__ __device__ inline uint64_t mix64(uint64_t x) {
  x ^= x >> 30;
  x *= 0xbf58476d1ce4e5b9ull;
  x ^= x >> 27;
  x *= 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}
__host__ __device__ inline uint64_t certificate(int B, int gmax, int V, uint32_t e) {
  uint64_t x = mix64(0x7376636572746966ull ^ (static_cast<uint64_t>(static_cast<uint32_t>(B)) << 32) ^
                     static_cast<uint32_t>(V));
  x = mix64(x ^ (static_cast<uint64_t>(static_cast<uint32_t>(gmax)) << 32) ^ e);
  return x | 1ull;
}

// Job flags and descriptor states carry the call's epoch: a value is current
// only if its tag matches, so neither array is ever reset between calls.
constexpr uint32_t kEpochMask = 0x3fffffffu;
__device__ __forceinline__ uint32_t epoch_tag(uint32_t e) { return (e & kEpochMask) << 2; }

// jflag[j] (with the call's tag): job j due / never due; any other value:
// not (yet) due.  Job b < B merges request b; job B + s searches the
// residual of descriptor slot s.
constexpr uint32_t kJobDue = 1u, kJobNone = 2u;
// An arrival count that marks a descriptor slot whose request turned out
// invalid (no residual, no search), for job warps that poll the counts.
constexpr uint32_t kSkipCount = 0xffffffffu;

// State of descriptor slot s (with the call's tag): holds a row to
// re-sample / holds nothing (its request turned out invalid); any other
// value: reserved but not yet written.
constexpr uint32_t kPending = 0u, kReadySample = 1u, kReadySkip = 2u;

// What a CTA knows of its call once the workspace header is checked.
struct Ctl {
  Counters *ctr;  // this call's counter set
  uint32_t *k1;   // [B] row-statistics chunks completed, this call's set
  uint32_t *k2;   // [B] residual chunks completed, this call's set
  uint32_t *err;  // this call's error word
  uint32_t tag;   // epoch_tag(epoch)
  uint32_t epoch;
  uint32_t ok;    // 0: the set could not be made clear (a fault); do no work
};

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
// field i in the low half of word i and the slot's tagged state in the high half.
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
// once every word carries it with the call's tag (d is then complete),
// kReadySkip as word 0 shows it, else kPending.
__device__ __forceinline__ uint32_t desc_poll(const uint64_t *w, Desc &d, uint32_t tag) {
  uint32_t *f = reinterpret_cast<uint32_t *>(&d);
  uint64_t v[kDescWords];
#pragma unroll
  for (int i = 0; i < kDescWords; ++i) v[i] = ld_relaxed64(w + i);
  const uint32_t s0 = static_cast<uint32_t>(v[0] >> 32);
  if (s0 == (tag | kReadySkip)) return kReadySkip;
  if (s0 != (tag | kReadySample)) return kPending;
  bool all = true;
#pragma unroll
  for (int i = 0; i < kDescWords; ++i) {
    all = all && static_cast<uint32_t>(v[i] >> 32) == (tag | kReadySample);
    f[i] = static_cast<uint32_t>(v[i]);
  }
  return all ? kReadySample : kPending;
}

// Waits (bounded) until every word of a kReadySample slot has landed.
__device__ __forceinline__ bool desc_read(const uint64_t *w, Desc &d, uint32_t tag,
                                          uint32_t *err) {
  uint32_t *f = reinterpret_cast<uint32_t *>(&d);
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint64_t v[kDescWords];
#pragma unroll
    for (int i = 0; i < kDescWords; ++i) v[i] = ld_relaxed64(w + i);
    bool all = true;
#pragma unroll
    for (int i = 0; i < kDescWords; ++i) {
      all = all && static_cast<uint32_t>(v[i] >> 32) == (tag | kReadySample);
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
  L.k1_cnt = take(sizeof(uint32_t) * 2 * B);  // one array per counter set
  L.k2_cnt = take(sizeof(uint32_t) * 2 * B);
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
  int tables_global;  // kernel 0 wrote row_start and cs (else each CTA builds them)
  int *row_start;    // [B+1] first flat row of each request (kernel 0)
  float *cs;         // [B] log2(e) / T, 0 for greedy (kernel 0)
  uint32_t *k1_cnt;  // [2][B] row-statistics chunks completed, per counter set
  uint32_t *k2_cnt;  // [2][B] residual chunks completed, per counter set
  uint64_t *desc;    // [B][kDescWords] rows to re-sample, in reservation (merge) order
  uint32_t *jflag;   // [2B] tagged kJobDue / kJobNone per job
  Part *part1;
  float2 *csum;      // [slot][C2] residual and p sums per chunk
  float2 *ssum;      // [slot][nseg] residual and p sums per 1024-element segment
};

// Warp-wide: clear counter set s (counters, per-request arrival counts and
// the set's error word) for a batch of B requests.
__device__ __forceinline__ void clear_set(const Params &p, int s, int lane) {
  uint32_t *c = reinterpret_cast<uint32_t *>(&p.hdr->set[s]);
  for (int i = lane; i < static_cast<int>(sizeof(Counters) / 4); i += 32) c[i] = 0u;
  uint32_t *k1 = p.k1_cnt + static_cast<size_t>(s) * p.B;
  uint32_t *k2 = p.k2_cnt + static_cast<size_t>(s) * p.B;
  for (int i = lane; i < p.B; i += 32) {
    k1[i] = 0u;
    k2[i] = 0u;
  }
  if (lane == 0) p.hdr->err[s] = 0u;
}

// Warp-wide: clear every job flag and descriptor word, so that no leftover
// value of a fresh or foreign workspace can carry a current tag.
__device__ __forceinline__ void clear_tags(const Params &p, int lane) {
  for (int i = lane; i < 2 * p.B; i += 32) p.jflag[i] = 0u;
  for (size_t i = lane; i < static_cast<size_t>(p.B) * kDescWords; i += 32) p.desc[i] = 0ull;
}

// Warp-wide: the call's counter set, from the header words the warp's lane
// 0 read after the grid dependency wait (epoch and error words, both
// certificates).  Set e & 1 serves the call with epoch e once its
// certificate says so; otherwise CTA 0 clears it (and every tag) while the
// other CTAs wait (bounded: on a timeout ok is 0 and nothing may use the
// set).  CTA 0 then clears the other set for the next call and certifies
// it.  Every CTA of the grid must be resident together.
__device__ __forceinline__ Ctl check_workspace(const Params &p, uint64_t hdr0, uint64_t rdy0,
                                               uint64_t rdy1, int lane, uint32_t *err) {
  const uint32_t e = static_cast<uint32_t>(__shfl_sync(kFull, static_cast<uint32_t>(hdr0), 0));
  const uint64_t r0 = __shfl_sync(kFull, rdy0, 0), r1 = __shfl_sync(kFull, rdy1, 0);
  const int s = static_cast<int>(e & 1u);
  const uint64_t key = certificate(p.B, p.gmax, p.V, e);
  const bool cta0 = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  bool ok = true;
  if ((s ? r1 : r0) != key) {
    if (cta0) {
      clear_set(p, s, lane);
      clear_tags(p, lane);
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        st_release64(&p.hdr->ready[s], key);
      }
    } else if (lane == 0) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire64(&p.hdr->ready[s]) != key) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicOr(err, SV_FAULT_TIMEOUT);
          ok = false;
          break;
        }
        __nanosleep(128);
      }
    }
    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
  }
  if (cta0) {
    clear_set(p, s ^ 1, lane);
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      st_release64(&p.hdr->ready[s ^ 1], certificate(p.B, p.gmax, p.V, e + 1u));
    }
  }
  Ctl c;
  c.ctr = &p.hdr->set[s];
  c.k1 = p.k1_cnt + static_cast<size_t>(s) * p.B;
  c.k2 = p.k2_cnt + static_cast<size_t>(s) * p.B;
  c.err = &p.hdr->err[s];
  c.tag = epoch_tag(e);
  c.epoch = e;
  c.ok = ok ? 1u : 0u;
  return c;
}

// The header words check_workspace needs (lane 0 of the checking warp).
__device__ __forceinline__ void read_header(const Params &p, uint64_t &hdr0, uint64_t &rdy0,
                                            uint64_t &rdy1) {
  hdr0 = ld_relaxed64(reinterpret_cast<const uint64_t *>(&p.hdr->epoch));
  rdy0 = ld_relaxed64(&p.hdr->ready[0]);
  rdy1 = ld_relaxed64(&p.hdr->ready[1]);
}

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
