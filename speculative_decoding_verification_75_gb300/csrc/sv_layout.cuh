// sv_layout.cuh -- workspace layout and launch parameters.
//
// The caller-owned workspace holds everything the three kernels hand to one
// another: per-request arrival counters, per-chunk partial statistics of the
// target softmax, the descriptors of the rows to be re-sampled and the
// per-chunk / per-segment residual sums that the inverse-CDF search walks.
#pragma once

#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>

#include "spec_verify.h"

namespace sv {

// Vocabulary tiling shared by every kernel.
constexpr int kSeg = 1024;              // elements per residual segment
constexpr int kK2Chunk = 4096;          // elements per re-sample chunk
constexpr int kMinChunk = 4096;         // smallest row-statistics chunk (fp32)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kQFloor = 1e-10f;       // clamp of the acceptance divisor

struct Header {                  // 256 bytes
  uint32_t err;                  // SV_BAD_* | SV_FAULT_* bits of this call
  uint32_t n_q;                  // re-sample descriptors that read a q row
  uint32_t n_noq;                // re-sample descriptors without a q row
  uint32_t k2_next;              // next re-sample item to hand out
  uint32_t pad[60];
};

struct __align__(8) Part {       // per (row, chunk) partial statistics
  float m;                       // chunk maximum logit
  float v;                       // sum exp2((l - m) * cs), or argmax bits
};

// Descriptor of one row to re-stream for the residual / bonus draw.
struct __align__(16) Desc {
  int b;                         // request
  int k;                         // first rejected position (g_b: bonus)
  int slot;                      // padded row index of row k
  int tok;                       // drafted token at k (one-hot q), or -1
  float m;                       // row maximum logit
  float inv_s;                   // 1 / normaliser
  float cs;                      // log2(e) / T
  float u;                       // sampling uniform
};

// Byte offsets of each region inside the workspace.
struct Layout {
  size_t hdr, k1_cnt, k2_cnt, desc_q, desc_noq, part1, csum, ssum, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

inline int div_up(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

inline Layout make_layout(int B, int gmax, int V) {
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(gmax + 1);
  const size_t c1 = static_cast<size_t>(div_up(V, kMinChunk));
  const size_t c2 = static_cast<size_t>(div_up(V, kK2Chunk));
  const size_t nseg = static_cast<size_t>(div_up(V, kSeg));
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.hdr = take(sizeof(Header));
  L.k1_cnt = take(sizeof(uint32_t) * B);
  L.k2_cnt = take(sizeof(uint32_t) * B);
  L.desc_q = take(sizeof(Desc) * B);
  L.desc_noq = take(sizeof(Desc) * B);
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
  int C;                         // row-statistics chunks per row (dtype dependent)
  int C2;                        // re-sample chunks per row
  int nseg;                      // residual segments per row
  int32_t *out_tokens;
  int32_t *out_nacc;
  sv_diag diag;
  Header *hdr;
  uint32_t *k1_cnt;
  uint32_t *k2_cnt;
  Desc *desc_q;
  Desc *desc_noq;
  Part *part1;
  float2 *csum;
  float2 *ssum;
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
