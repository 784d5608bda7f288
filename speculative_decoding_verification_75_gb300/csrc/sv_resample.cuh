// sv_resample.cuh -- the residual (or bonus) sums of one chunk, and the
// inverse-CDF search of a request.
//
// Tutorial page dpshk.com/news/5598276 (HTML title 企业官网建设流程全解析):
// §3.1 step 4 and §5.2 step (5) (_recover_rejected): r = (p_k - q_k)_+,
// normalised, sampled once; §5.3: the bonus token is drawn from p_g.  The
// page's multinomial draw becomes an inverse-CDF draw on the caller's uniform:
// token = min{ j : C_j > u * S }, C the inclusive prefix sum of r, S = C_V.
//
// Only the row each sampled request draws from is re-read, and q only at a
// rejection.  A consumer warp forms p and (p - q)_+ on the fly with packed
// fp32x2 arithmetic and records the sums of every 1024-element segment; when
// every chunk of the request is done, one warp walks chunk sums, segment sums
// and then the elements of one segment to find the token: a three-level
// search that re-reads 1024 elements instead of the whole row.
#pragma once

#include "sv_device.cuh"
#include "sv_layout.cuh"

namespace sv {

// p_j of the target softmax and r_j = (p_j - q_j)_+, as a fixed sequence of
// correctly rounded operations: the packed fp32x2 forms in the streaming pass
// and these scalar forms in the search give identical values.
// p(x) = exp2(x * cs - o) / s, with o = fl(m * cs) for the row maximum m and
// s the row's sum relative to the same offset (the merge keeps it so).
__device__ __forceinline__ float target_p(float x, float nego, float cs, float inv_s) {
  return __fmul_rn(ex2(__fmaf_rn(x, cs, nego)), inv_s);
}
__device__ __forceinline__ float resid(float p, float q) {
  return fmaxf(__fsub_rn(p, q), 0.f);
}
__device__ __forceinline__ float2 target_p2(float2 x, float2 nego, float2 cs2, float2 inv2) {
  const float2 t = __ffma2_rn(x, cs2, nego);
  return __fmul2_rn(make_float2(ex2(t.x), ex2(t.y)), inv2);
}

// ------------------------------------------------------------ search ----

// One level of the inverse-CDF walk over n <= 64 weights held two per lane
// (w0 for index lane, w1 for lane + 32), starting at `carry`: the first index
// with positive weight whose inclusive prefix exceeds target, else the last
// index with positive weight (then *fell_back is set).  Also returns the
// exclusive prefix.
__device__ __forceinline__ int cdf_level64(int n, float w0, float w1, float carry,
                                           float target, int lane, float *excl_out,
                                           bool *fell_back) {
  int last = -1;
  float last_excl = carry;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = 32 * r + lane;
    const float w = (i < n) ? (r ? w1 : w0) : 0.f;
    const float incl = carry + warp_inclusive_scan(w, lane);
    const float prev = __shfl_up_sync(kFull, incl, 1);
    const float excl = (lane == 0) ? carry : prev;
    const unsigned hit = __ballot_sync(kFull, i < n && w > 0.f && incl > target);
    if (hit) {
      const int src = __ffs(hit) - 1;
      *excl_out = __shfl_sync(kFull, excl, src);
      return 32 * r + src;
    }
    const unsigned pos = __ballot_sync(kFull, i < n && w > 0.f);
    if (pos) {
      const int src = 31 - __clz(pos);
      last = 32 * r + src;
      last_excl = __shfl_sync(kFull, excl, src);
    }
    carry = __shfl_sync(kFull, incl, 31);
  }
  *excl_out = last_excl;
  *fell_back = true;
  return last;
}

// Generic level for any n: rounds of 32 weights fetched by `weight`.
template <typename W>
__device__ __forceinline__ int cdf_level(int n, float carry, float target, int lane,
                                         W weight, float *excl_out, bool *fell_back) {
  int last = -1;
  float last_excl = carry;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const float w = (i < n) ? weight(i) : 0.f;
    const float incl = carry + warp_inclusive_scan(w, lane);
    const float prev = __shfl_up_sync(kFull, incl, 1);
    const float excl = (lane == 0) ? carry : prev;
    const unsigned hit = __ballot_sync(kFull, i < n && w > 0.f && incl > target);
    if (hit) {
      const int src = __ffs(hit) - 1;
      *excl_out = __shfl_sync(kFull, excl, src);
      return i0 + src;
    }
    const unsigned pos = __ballot_sync(kFull, i < n && w > 0.f);
    if (pos) {
      const int src = 31 - __clz(pos);
      last = i0 + src;
      last_excl = __shfl_sync(kFull, excl, src);
    }
    carry = __shfl_sync(kFull, incl, 31);
  }
  *excl_out = last_excl;
  *fell_back = true;
  return last;
}

// The q value the draw subtracts at element j (before the clamp at 0).
__device__ __forceinline__ float q_at(const Params &p, const Desc &d, int j) {
  if (d.tok < 0) return 0.f;                        // bonus row: nothing
  if (p.q) return __ldg(p.q + (static_cast<size_t>(d.b) * p.gmax + d.k) * p.V + j);
  return (j == d.tok) ? 1.f : 0.f;                  // deterministic draft
}

// Element level over one segment of n <= 1024 elements starting at e0: lane
// l owns elements 32l..32l+31 and loads all of them at once (16-byte vectors
// when the row is aligned); the lanes' totals are scanned to give each lane
// its starting prefix.
template <typename T, bool kVec>
__device__ __forceinline__ int search_segment(const Params &p, const Desc &d, int e0, int n,
                                              float carry, float target, bool use_p,
                                              int lane) {
  const T *row = static_cast<const T *>(p.logits) + static_cast<size_t>(d.slot) * p.V;
  const float nego = -__fmul_rn(d.m, d.cs);  // the row's exponent offset, negated
  const int l0 = 32 * lane;
  float x[32], q[32];
  if (kVec && l0 + 32 <= n) {
    if constexpr (sizeof(T) == 2) {
      const uint4 *src = reinterpret_cast<const uint4 *>(row + e0 + l0);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 w = __ldg(src + v);
        x[8 * v + 0] = bf16_lo(w.x); x[8 * v + 1] = bf16_hi(w.x);
        x[8 * v + 2] = bf16_lo(w.y); x[8 * v + 3] = bf16_hi(w.y);
        x[8 * v + 4] = bf16_lo(w.z); x[8 * v + 5] = bf16_hi(w.z);
        x[8 * v + 6] = bf16_lo(w.w); x[8 * v + 7] = bf16_hi(w.w);
      }
    } else {
      const float4 *src = reinterpret_cast<const float4 *>(row + e0 + l0);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 w = __ldg(src + v);
        x[4 * v + 0] = w.x; x[4 * v + 1] = w.y; x[4 * v + 2] = w.z; x[4 * v + 3] = w.w;
      }
    }
    if (d.tok >= 0 && p.q) {
      const float4 *qs = reinterpret_cast<const float4 *>(
          p.q + (static_cast<size_t>(d.b) * p.gmax + d.k) * p.V + e0 + l0);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 w = __ldg(qs + v);
        q[4 * v + 0] = w.x; q[4 * v + 1] = w.y; q[4 * v + 2] = w.z; q[4 * v + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int t = 0; t < 32; ++t) q[t] = (d.tok >= 0 && e0 + l0 + t == d.tok) ? 1.f : 0.f;
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const bool in = l0 + t < n;
      x[t] = in ? Elem<T>::load(row, e0 + l0 + t) : -INFINITY;
      q[t] = in ? q_at(p, d, e0 + l0 + t) : 0.f;
    }
  }
  float w[32];
  float tot = 0.f;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const float pj = target_p(x[t], nego, d.cs, d.inv_s);
    w[t] = (l0 + t < n) ? (use_p ? pj : resid(pj, q[t])) : 0.f;
    tot += w[t];
  }
  const float incl = carry + warp_inclusive_scan(tot, lane);
  const float prev = __shfl_up_sync(kFull, incl, 1);
  float c = (lane == 0) ? carry : prev;
  int hit = -1, lastpos = -1;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    c += w[t];
    if (hit < 0 && w[t] > 0.f && c > target) hit = t;
    if (w[t] > 0.f) lastpos = t;
  }
  const unsigned hb = __ballot_sync(kFull, hit >= 0);
  if (hb) {
    const int src = __ffs(hb) - 1;
    return e0 + 32 * src + __shfl_sync(kFull, hit, src);
  }
  // Rounding left u*S at or past the total: the last positive weight.
  const unsigned pb = __ballot_sync(kFull, lastpos >= 0);
  if (!pb) return e0;
  const int src = 31 - __clz(pb);
  return e0 + 32 * src + __shfl_sync(kFull, lastpos, src);
}

// Inverse-CDF walk over n <= 256 weights held eight per lane, lane l owning
// indices 8l..8l+7 in order: the first index with positive weight whose
// inclusive prefix exceeds target, else the last index with positive weight
// (then *fell_back is set).  Also returns the exclusive prefix at that index.
// Every level of the draw skips zero weights this way: with u * S within
// rounding of the total, a scanned prefix can pass the target at an index
// that holds nothing (a padded lane past the end of the row included).
__device__ __forceinline__ int cdf_block8(int n, const float (&w)[8], float target, int lane,
                                          float *excl_out, bool *fell_back) {
  float tot = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) tot += (8 * lane + j < n) ? w[j] : 0.f;
  const float incl = warp_inclusive_scan(tot, lane);
  const float prev = __shfl_up_sync(kFull, incl, 1);
  float c = (lane == 0) ? 0.f : prev;  // this lane's starting prefix
  int hit = -1, lastpos = -1;
  float hit_excl = 0.f, last_excl = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool in = 8 * lane + j < n;
    const float wj = in ? w[j] : 0.f;
    if (in && hit < 0 && wj > 0.f && c + wj > target) {
      hit = j;
      hit_excl = c;
    }
    if (in && wj > 0.f) {
      lastpos = j;
      last_excl = c;
    }
    c += wj;
  }
  const unsigned hb = __ballot_sync(kFull, hit >= 0);
  if (hb) {
    const int src = __ffs(hb) - 1;
    *excl_out = __shfl_sync(kFull, hit_excl, src);
    return 8 * src + __shfl_sync(kFull, hit, src);
  }
  *fell_back = true;
  const unsigned pb = __ballot_sync(kFull, lastpos >= 0);
  if (!pb) {
    *excl_out = 0.f;
    return -1;
  }
  const int src = 31 - __clz(pb);
  *excl_out = __shfl_sync(kFull, last_excl, src);
  return 8 * src + __shfl_sync(kFull, lastpos, src);
}

// Draw of descriptor slot sl (row d), once every chunk of its residual is
// reduced.  Rows of up to 256 segments: one wave of loads fetches every
// segment sum, a walk over them finds the segment, a second wave fetches its
// elements.  Longer rows walk chunk sums, segment sums, then elements.
// Warp-wide: slot sl's descriptor, read (and waited for) by lane 0 and handed
// to every lane; false if the wait gave up.
__device__ __forceinline__ bool desc_read_warp(const Params &p, const Ctl &c, int sl, int lane,
                                               Desc &d) {
  bool ok = true;
  if (lane == 0) ok = desc_read(p.desc + static_cast<size_t>(sl) * kDescWords, d, c.tag, c.err);
  if (!__shfl_sync(kFull, ok ? 1 : 0, 0)) return false;
  uint32_t *f = reinterpret_cast<uint32_t *>(&d);
#pragma unroll
  for (int i = 0; i < kDescWords; ++i) f[i] = __shfl_sync(kFull, f[i], 0);
  return true;
}

// The search of slot sl.  The segment sums depend on the slot alone, so
// their loads go out before the descriptor is read: both round trips overlap.
template <typename T, bool kVec>
__device__ __noinline__ void search_request(const Params &p, const Ctl ctl, int sl, int lane) {
  const float2 *cs2 = p.csum + static_cast<size_t>(sl) * p.C2;
  const float2 *ss2 = p.ssum + static_cast<size_t>(sl) * p.nseg;
  const int nsr = (p.V + kSeg - 1) / kSeg;  // segments of the row
  Desc d{};
  if (nsr <= 256) {
    float wr[8], wp[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = 8 * lane + j;
      const float2 v = (i < nsr) ? ld_cg(ss2 + i) : make_float2(0.f, 0.f);
      wr[j] = v.x;
      wp[j] = v.y;
    }
    if (!desc_read_warp(p, ctl, sl, lane, d)) return;
    float lr = 0.f, lp = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      lr += wr[j];
      lp += wp[j];
    }
    const float tr = __shfl_sync(kFull, warp_inclusive_scan(lr, lane), 31);
    const float tp = __shfl_sync(kFull, warp_inclusive_scan(lp, lane), 31);
    const bool use_p = !(tr > 0.f);  // empty residual: draw from p itself
    float target = __fmul_rn(d.u, use_p ? tp : tr);
    bool fb = false;
    float base = 0.f;
    const int sg = max(0, cdf_block8(nsr, use_p ? wp : wr, target, lane, &base, &fb));
    if (fb) target = INFINITY;  // rounding pushed u*S past the total
    const int j = search_segment<T, kVec>(p, d, sg * kSeg, min(kSeg, p.V - sg * kSeg), base,
                                          target, use_p, lane);
    if (lane == 0) {
      p.out_tokens[static_cast<size_t>(d.b) * (p.gmax + 1) + d.k] = j;
      if (p.diag.resid_mass) p.diag.resid_mass[d.b] = tr;
    }
    return;
  }

  if (!desc_read_warp(p, ctl, sl, lane, d)) return;
  // Totals of the residual and of p, in the same scan order the walk uses.
  float tr = 0.f, tp = 0.f;
  float2 v0 = make_float2(0.f, 0.f), v1 = v0;
  const bool small = p.C2 <= 64;
  if (small) {
    if (lane < p.C2) v0 = ld_cg(cs2 + lane);
    if (lane + 32 < p.C2) v1 = ld_cg(cs2 + lane + 32);
    tr = __shfl_sync(kFull, warp_inclusive_scan(v0.x, lane), 31);
    tp = __shfl_sync(kFull, warp_inclusive_scan(v0.y, lane), 31);
    tr = __shfl_sync(kFull, tr + warp_inclusive_scan(v1.x, lane), 31);
    tp = __shfl_sync(kFull, tp + warp_inclusive_scan(v1.y, lane), 31);
  } else {
    for (int c0 = 0; c0 < p.C2; c0 += 32) {
      const int c = c0 + lane;
      const float2 v = (c < p.C2) ? ld_cg(cs2 + c) : make_float2(0.f, 0.f);
      tr = __shfl_sync(kFull, tr + warp_inclusive_scan(v.x, lane), 31);
      tp = __shfl_sync(kFull, tp + warp_inclusive_scan(v.y, lane), 31);
    }
  }
  const bool use_p = !(tr > 0.f);  // empty residual: draw from p itself
  const float S = use_p ? tp : tr;
  float target = __fmul_rn(d.u, S);
  bool fb = false;

  // Each level returns a valid index whenever its weights have a positive
  // total (validated inputs guarantee it); the clamps only keep pathological
  // caller data (e.g. -inf draft probabilities) inside the row.
  float base = 0.f;
  int c;
  if (small) {
    c = cdf_level64(p.C2, use_p ? v0.y : v0.x, use_p ? v1.y : v1.x, 0.f, target, lane,
                    &base, &fb);
  } else {
    c = cdf_level(
        p.C2, 0.f, target, lane,
        [&](int i) { const float2 v = ld_cg(cs2 + i); return use_p ? v.y : v.x; }, &base,
        &fb);
  }
  c = max(0, c);
  if (fb) target = INFINITY;  // rounding pushed u*S past the total
  constexpr int kChunk = Tiling<T>::kResChunk;
  const int g0 = c * Tiling<T>::kSegPerChunk;
  const int nsg = (min(kChunk, p.V - c * kChunk) + kSeg - 1) / kSeg;
  float2 sv = make_float2(0.f, 0.f);
  if (lane < nsg) sv = ld_cg(ss2 + g0 + lane);
  float base2 = 0.f;
  const int sg = g0 + max(0, cdf_level64(nsg, use_p ? sv.y : sv.x, 0.f, base, target, lane,
                                         &base2, &fb));
  if (fb) target = INFINITY;
  const int j = search_segment<T, kVec>(p, d, sg * kSeg, min(kSeg, p.V - sg * kSeg), base2,
                                        target, use_p, lane);
  if (lane == 0) {
    p.out_tokens[static_cast<size_t>(d.b) * (p.gmax + 1) + d.k] = j;
    if (p.diag.resid_mass) p.diag.resid_mass[d.b] = tr;
  }
}

// ------------------------------------------------------ chunk residual ----

// Residual and p sums of one chunk per 1024-element segment, for the
// segments h, h + 2, ... of the chunk (two warps share a chunk).  Writes the
// segment sums and returns this warp's share of the chunk sums (in lane 0).
// Lane layout: each 256-element step gives lane l the elements 4l..4l+3 and
// 128+4l..128+4l+3 (conflict-free 8- and 16-byte shared-memory reads).
template <typename T, bool kTMA>
__device__ __forceinline__ float2 chunk_resid(const Params &p, const Desc &d, int sl, int chunk,
                                              int ne, bool has_q, const uint8_t *stage, int h,
                                              int lane) {
  constexpr int kChunk = Tiling<T>::kResChunk;
  const int e0 = chunk * kChunk;
  const T *row = static_cast<const T *>(p.logits) + static_cast<size_t>(d.slot) * p.V;
  const float *qrow =
      has_q ? p.q + (static_cast<size_t>(d.b) * p.gmax + d.k) * p.V : nullptr;
  const float *sq = reinterpret_cast<const float *>(stage + kChunk * sizeof(T));
  const float nego1 = -__fmul_rn(d.m, d.cs);  // the row's exponent offset, negated
  const float2 nego = make_float2(nego1, nego1), cs2 = make_float2(d.cs, d.cs);
  const float2 inv2 = make_float2(d.inv_s, d.inv_s), zero2 = make_float2(0.f, 0.f);
  const bool onehot = d.tok >= 0 && !has_q;
  const int nsg = (ne + kSeg - 1) / kSeg;
  float chunk_r = 0.f, chunk_p = 0.f;
  for (int sgi = h; sgi < nsg; sgi += 2) {
    float2 ar = zero2, ap = zero2;
#pragma unroll
    for (int step = 0; step < kSeg / 256; ++step) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int e = sgi * kSeg + step * 256 + half * 128 + 4 * lane;  // in chunk
        if (e < ne) {
          float2 x01, x23, q01 = zero2, q23 = zero2;  // q held negated
          if (kTMA) {
            if constexpr (sizeof(T) == 2) {
              const uint2 w = *reinterpret_cast<const uint2 *>(stage + 2 * e);
              x01 = make_float2(bf16_lo(w.x), bf16_hi(w.x));
              x23 = make_float2(bf16_lo(w.y), bf16_hi(w.y));
            } else {
              const float4 w = *reinterpret_cast<const float4 *>(stage + 4 * e);
              x01 = make_float2(w.x, w.y);
              x23 = make_float2(w.z, w.w);
            }
            if (has_q) {
              const float4 w = *reinterpret_cast<const float4 *>(sq + e);
              q01 = make_float2(-w.x, -w.y);
              q23 = make_float2(-w.z, -w.w);
            }
          } else {
            float xs[4], qs[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              // elements past the chunk end weigh nothing (p = q = 0 there)
              const bool in = e + t < ne;
              xs[t] = in ? Elem<T>::load(row, e0 + e + t) : -INFINITY;
              qs[t] = (in && qrow) ? -__ldg(qrow + e0 + e + t) : 0.f;
            }
            x01 = make_float2(xs[0], xs[1]);
            x23 = make_float2(xs[2], xs[3]);
            q01 = make_float2(qs[0], qs[1]);
            q23 = make_float2(qs[2], qs[3]);
          }
          const float2 p01 = target_p2(x01, nego, cs2, inv2);
          const float2 p23 = target_p2(x23, nego, cs2, inv2);
          const float2 d01 = __fadd2_rn(p01, q01), d23 = __fadd2_rn(p23, q23);
          float r[4] = {fmaxf(d01.x, 0.f), fmaxf(d01.y, 0.f), fmaxf(d23.x, 0.f),
                        fmaxf(d23.y, 0.f)};
          if (onehot) {
            const unsigned off = static_cast<unsigned>(d.tok - (e0 + e));
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (off == static_cast<unsigned>(t)) r[t] = 0.f;  // (p - 1)_+ = 0
          }
          ar = __fadd2_rn(ar, make_float2(r[0], r[1]));
          ar = __fadd2_rn(ar, make_float2(r[2], r[3]));
          ap = __fadd2_rn(ap, p01);
          ap = __fadd2_rn(ap, p23);
        }
      }
    }
    const float sr = warp_sum(ar.x + ar.y);
    const float sp = warp_sum(ap.x + ap.y);
    if (lane == 0) {
      p.ssum[static_cast<size_t>(sl) * p.nseg + chunk * Tiling<T>::kSegPerChunk + sgi] =
          make_float2(sr, sp);
      chunk_r += sr;
      chunk_p += sp;
    }
  }
  return make_float2(chunk_r, chunk_p);
}

}  // namespace sv
