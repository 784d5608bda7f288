// sv_rowstats.cuh -- target-softmax statistics of one vocabulary chunk, and
// the merge + accept step of a request.
//
// Tutorial page dpshk.com/news/5598276 (HTML title 企业官网建设流程全解析),
// §5.2 steps (1)-(4): softmax of the g+1 target rows, a_i = min(1, p/q) with
// q clamped at 1e-10, accepted = u < a, cumprod prefix = first rejection.
//
// A consumer warp reduces one chunk held in shared memory: pass A takes the
// maximum m (packed bf16x2 max), pass B the sum of exp2(l * cs - o) with
// cs = log2(e)/T and the offset o = fl(m * cs), one packed fp32x2 fma per
// pair of logits (greedy rows instead find the lowest index of the maximum).
// The fma forms l * cs - o exactly and rounds once, so each exponent is
// accurate relative to its own size, and whoever combines the statistics
// recomputes o from m: the sum stands for exp2((l - m) * cs) summed, times
// the exact factor exp2(m * cs - o).  p itself is never stored: only (max, sum) per chunk reaches
// global memory.  When every chunk of a request is done, one warp merges the
// chunk statistics in chunk order, checks the request's inputs, gathers
// p(x_i) and q(x_i), runs the accept test for all positions with one ballot,
// writes the accepted drafts and publishes the row to re-sample.
#pragma once

#include "sv_device.cuh"
#include "sv_layout.cuh"

namespace sv {

// ------------------------------------------------- chunk statistics ----

struct ChunkStat {
  float m;  // maximum logit of the chunk
  float v;  // sum of exp2(l * cs - offset(m, cs)), or the argmax bits for greedy rows
};

// The exponent offset of a chunk (or row) whose maximum is m.
__device__ __forceinline__ float offset(float m, float cs) { return __fmul_rn(m, cs); }

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162 *>(&a),
                             *reinterpret_cast<__nv_bfloat162 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// exp2(x * cs - o) for a pair (nego = -o), one packed fp32x2 fma.
__device__ __forceinline__ float2 exp_pair(float2 x, float2 nego, float2 cs2) {
  const float2 t = __ffma2_rn(x, cs2, nego);
  return make_float2(ex2(t.x), ex2(t.y));
}

// bf16 chunk staged in shared memory; ne is a multiple of 8.
__device__ __forceinline__ ChunkStat chunk_stats_smem(const __nv_bfloat16 *stage,
                                                      int ne, float cs, int lane) {
  const uint4 *v = reinterpret_cast<const uint4 *>(stage);
  const int nvec = ne >> 3;
  uint32_t mx = 0xff80ff80u;  // (-inf, -inf)
#pragma unroll 4
  for (int i = lane; i < nvec; i += 32) {
    const uint4 x = v[i];
    mx = bmax2(mx, bmax2(bmax2(x.x, x.y), bmax2(x.z, x.w)));
  }
  const float m = warp_max(fmaxf(bf16_lo(mx), bf16_hi(mx)));
  ChunkStat r{m, 0.f};
  if (cs != 0.f) {
    if (m == -INFINITY) return r;  // fully masked chunk contributes nothing
    const float o = offset(m, cs);
    const float2 nego = make_float2(-o, -o), cs2 = make_float2(cs, cs);
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll 4
    for (int i = lane; i < nvec; i += 32) {
      const uint4 x = v[i];
      a0 = __fadd2_rn(a0, exp_pair(make_float2(bf16_lo(x.x), bf16_hi(x.x)), nego, cs2));
      a1 = __fadd2_rn(a1, exp_pair(make_float2(bf16_lo(x.y), bf16_hi(x.y)), nego, cs2));
      a0 = __fadd2_rn(a0, exp_pair(make_float2(bf16_lo(x.z), bf16_hi(x.z)), nego, cs2));
      a1 = __fadd2_rn(a1, exp_pair(make_float2(bf16_lo(x.w), bf16_hi(x.w)), nego, cs2));
    }
    r.v = warp_sum((a0.x + a0.y) + (a1.x + a1.y));
    return r;
  }
  // Greedy row: lowest index holding the maximum.  Each 32-vector step covers
  // 256 consecutive elements, so the first step with a hit holds the answer.
  int found = 0x7fffffff;
  for (int base = 0; base < nvec; base += 32) {
    const int i = base + lane;
    int hit = 8;
    if (i < nvec) {
      const uint4 x = v[i];
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        const float e = (j & 1) ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1]);
        if (e == m) hit = j;
      }
    }
    const unsigned bal = __ballot_sync(kFull, hit < 8);
    if (bal) {
      const int src = __ffs(bal) - 1;
      found = (base + src) * 8 + __shfl_sync(kFull, hit, src);
      break;
    }
  }
  r.v = __int_as_float(found);
  return r;
}

// fp32 chunk staged in shared memory; ne is a multiple of 4.
__device__ __forceinline__ ChunkStat chunk_stats_smem(const float *stage, int ne,
                                                      float cs, int lane) {
  const float4 *v = reinterpret_cast<const float4 *>(stage);
  const int nvec = ne >> 2;
  float mx = -INFINITY;
#pragma unroll 4
  for (int i = lane; i < nvec; i += 32) {
    const float4 x = v[i];
    mx = fmaxf(mx, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
  }
  const float m = warp_max(mx);
  ChunkStat r{m, 0.f};
  if (cs != 0.f) {
    if (m == -INFINITY) return r;
    const float o = offset(m, cs);
    const float2 nego = make_float2(-o, -o), cs2 = make_float2(cs, cs);
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll 4
    for (int i = lane; i < nvec; i += 32) {
      const float4 x = v[i];
      a0 = __fadd2_rn(a0, exp_pair(make_float2(x.x, x.y), nego, cs2));
      a1 = __fadd2_rn(a1, exp_pair(make_float2(x.z, x.w), nego, cs2));
    }
    r.v = warp_sum((a0.x + a0.y) + (a1.x + a1.y));
    return r;
  }
  int found = 0x7fffffff;
  for (int base = 0; base < nvec; base += 32) {
    const int i = base + lane;
    int hit = 4;
    if (i < nvec) {
      const float4 x = v[i];
      if (x.w == m) hit = 3;
      if (x.z == m) hit = 2;
      if (x.y == m) hit = 1;
      if (x.x == m) hit = 0;
    }
    const unsigned bal = __ballot_sync(kFull, hit < 4);
    if (bal) {
      const int src = __ffs(bal) - 1;
      found = (base + src) * 4 + __shfl_sync(kFull, hit, src);
      break;
    }
  }
  r.v = __int_as_float(found);
  return r;
}

// Any dtype, any alignment: direct element loads from global memory.
template <typename T>
__device__ __forceinline__ ChunkStat chunk_stats_global(const T *row, int e0, int ne,
                                                        float cs, int lane) {
  float mx = -INFINITY;
  for (int j = lane; j < ne; j += 32) mx = fmaxf(mx, Elem<T>::load(row, e0 + j));
  const float m = warp_max(mx);
  ChunkStat r{m, 0.f};
  if (cs != 0.f) {
    if (m == -INFINITY) return r;
    const float o = offset(m, cs);
    float s = 0.f;
    for (int j = lane; j < ne; j += 32) s += ex2(__fmaf_rn(Elem<T>::load(row, e0 + j), cs, -o));
    r.v = warp_sum(s);
    return r;
  }
  int found = 0x7fffffff;
  for (int base = 0; base < ne; base += 32) {
    const int j = base + lane;
    const bool hit = j < ne && Elem<T>::load(row, e0 + j) == m;
    const unsigned bal = __ballot_sync(kFull, hit);
    if (bal) {
      found = base + __ffs(bal) - 1;
      break;
    }
  }
  r.v = __int_as_float(found);
  return r;
}

// A part's sum v scaled to another offset by scale = exp2(offset difference).
// A zero scale wins over an infinite v: a part whose maximum lies so far
// below the row's that its weight underflows adds nothing, even when its
// own sum overflowed (the rounding error of its offset, m_c * cs, can exceed
// the binary32 exponent range once |m_c * cs| >= 2^31, for valid rows with
// a tiny T).  A NaN sum (a NaN logit) still propagates.
__device__ __forceinline__ float scaled_part(float v, float scale) {
  return (scale == 0.f && !isnan(v)) ? 0.f : __fmul_rn(v, scale);
}

// Largest |m * cs| (row maximum in log2 units) for which the step can form
// its exponents in binary32: beyond it the rounding error of m * cs alone
// exceeds 1, and the row is invalid data.
constexpr float kExpLimit = 16777216.f;  // 2^24

// Two warps share a chunk: half 0 takes the first ne0 elements (a multiple
// of 8, at least half), half 1 the rest.
__device__ __forceinline__ int half0_len(int ne) { return min(ne, ((ne + 15) >> 4) << 3); }

// Statistics of a chunk from those of its two halves (half 1 follows half
// 0).  Greedy rows keep the lowest index of the maximum.
__device__ __forceinline__ ChunkStat combine_halves(ChunkStat a, ChunkStat b, float cs) {
  if (cs == 0.f) return (b.m > a.m) ? b : a;
  const float m = fmaxf(a.m, b.m), o = offset(m, cs);
  float s = 0.f;
  if (a.m != -INFINITY) s = scaled_part(a.v, ex2(__fsub_rn(offset(a.m, cs), o)));
  if (b.m != -INFINITY) s = __fadd_rn(s, scaled_part(b.v, ex2(__fsub_rn(offset(b.m, cs), o))));
  return ChunkStat{m, s};
}

// ----------------------------------------------------- merge + accept ----

// Counts a finished merge (after its reservation and flags); the last one
// raises all_merged, after which b_reserved is final for whoever acquires
// the flag.
__device__ __forceinline__ void count_merged(const Params &p, const Ctl &c) {
  if (atomic_add_acq_rel(&c.ctr->n_merged, 1u) + 1u == static_cast<uint32_t>(p.B))
    st_release(&c.ctr->all_merged, 1u);
}

// Outputs of a request whose draft length is invalid (it has no rows): -1
// tokens and num_accepted, NaN / flag 2 diagnostics; counted as finished.
__device__ void fill_bad_request(const Params &p, const Ctl &c, int b) {
  const int R = p.gmax + 1;
  const float qnan = __int_as_float(0x7fc00000);
  for (int i = 0; i < R; ++i) p.out_tokens[static_cast<size_t>(b) * R + i] = -1;
  p.out_nacc[b] = -1;
  const sv_diag &d = p.diag;
  for (int i = 0; i < p.gmax; ++i) {
    const size_t pi = static_cast<size_t>(b) * p.gmax + i;
    if (d.p_tok) d.p_tok[pi] = qnan;
    if (d.q_tok) d.q_tok[pi] = qnan;
    if (d.accept_prob) d.accept_prob[pi] = qnan;
    if (d.flags) d.flags[pi] = 2;
  }
  for (int i = 0; i < R; ++i) {
    const size_t ri = static_cast<size_t>(b) * R + i;
    if (d.row_max) d.row_max[ri] = qnan;
    if (d.row_sum) d.row_sum[ri] = qnan;
    if (d.row_argmax) d.row_argmax[ri] = -1;
  }
  if (d.resid_mass) d.resid_mass[b] = qnan;
  atomicOr(c.err, SV_BAD_DRAFT_LEN);
  if (d.accept_hist) atomicAdd(d.accept_hist + p.gmax + 1, 1);
  count_merged(p, c);
}

constexpr int kMergeBatch = 16;

// The inputs of draft position i of request b that the accept test reads:
// the drafted token x, its uniform u, the target logit at x and q_i(x)
// (loaded only where they are used; an out-of-range x reads entry 0 and is
// flagged by the merge).
struct DraftIn {
  int x;
  float u, lx, q;
};

template <typename T>
__device__ __forceinline__ DraftIn load_draft_inputs(const Params &p, int b, int g, bool greedy,
                                                     int i) {
  const bool draft = i < g;
  const size_t pi = static_cast<size_t>(b) * p.gmax + (draft ? i : 0);
  DraftIn d;
  d.x = draft ? __ldg(p.ids + pi) : 0;
  d.u = draft ? __ldg(p.u_acc + pi) : 0.f;
  const int xc = (d.x >= 0 && d.x < p.V) ? d.x : 0;
  d.lx = (draft && !greedy)
             ? Elem<T>::load(static_cast<const T *>(p.logits),
                             (static_cast<size_t>(b) * (p.gmax + 1) + i) * p.V + xc)
             : 0.f;
  d.q = (draft && p.q) ? __ldg(p.q + pi * p.V + xc) : 1.f;
  return d;
}

// The state of a request's accept step, carried across its groups of 32 rows.
struct Decision {
  int k = -1;                 // first rejected position
  float mk = 0.f, sk = 1.f;   // its row statistics
  int ak = -1, xk = -1;       // its argmax and drafted token
  float mg = 0.f, sg = 1.f;   // bonus row statistics
  int ag = -1;
  int x0 = 0;                 // this lane's draft id in the first group
  uint32_t bad = 0;
};

// Folds a batch of n <= kMergeBatch partial statistics (maximum, sum
// relative to that maximum's offset; -inf maximum: empty) into the running
// pair (m, s): the batch's maximum first, then its sums against that offset
// as independent terms, then the batch into the running pair.  Greedy rows
// (cs = 0) keep the first maximum and its argmax bits instead.
__device__ __forceinline__ void fold_batch(const Part (&q)[kMergeBatch], int n, float cs,
                                           float &m, float &s, int &am) {
  if (cs == 0.f) {
#pragma unroll
    for (int tj = 0; tj < kMergeBatch; ++tj) {
      if (tj >= n) break;
      if (q[tj].m > m || am < 0) {
        m = q[tj].m;
        am = __float_as_int(q[tj].v);
      }
    }
    return;
  }
  float bm = -INFINITY;
#pragma unroll
  for (int tj = 0; tj < kMergeBatch; ++tj) bm = fmaxf(bm, q[tj].m);  // padding is -inf
  if (bm == -INFINITY) return;  // every part of the batch empty
  const float ob = offset(bm, cs);
  float bs = 0.f;
#pragma unroll
  for (int tj = 0; tj < kMergeBatch; ++tj)
    if (q[tj].m != -INFINITY)
      bs = __fadd_rn(bs, scaled_part(q[tj].v, ex2(__fsub_rn(offset(q[tj].m, cs), ob))));
  if (bm > m) {
    s = __fadd_rn(scaled_part(s, ex2(__fsub_rn(offset(m, cs), ob))), bs);
    m = bm;
  } else {
    s = __fadd_rn(s, scaled_part(bs, ex2(__fsub_rn(ob, offset(m, cs)))));
  }
}

// Warp-wide accept step of rows i0 .. i0+31 of request b (nr rows, the last
// the bonus row).  Lane i - i0 holds row i's statistics -- maximum m, sum s
// relative to offset(m), lowest argmax am (greedy) -- and, for a draft
// position, its inputs.  Checks the inputs, writes the row's and position's
// diagnostics (unless out is false: a peer computing the same decision),
// runs the accept test and records the first rejection and the bonus row in
// dc.
__device__ __forceinline__ void accept_group(const Params &p, int b, int nr, float cs, int i0,
                                             int lane, float m, float s, int am,
                                             const DraftIn &in, Decision &dc, bool out = true) {
  const int g = nr - 1;
  const int R = p.gmax + 1;
  const bool greedy = (cs == 0.f);
  const sv_diag dg = out ? p.diag : sv_diag{};
  const int i = i0 + lane;
  const bool row = i < nr, draft = i < g;
  const size_t pi = static_cast<size_t>(b) * p.gmax + (draft ? i : 0);
  const int x = in.x;
  const float u = in.u, lx = in.lx, qraw = in.q;
  const bool x_ok = x >= 0 && x < p.V;
  const int xc = x_ok ? x : 0;
  if (i0 == 0) dc.x0 = x;
  bool f = true;
  if (row) {
    if (draft) {
      if (!x_ok) dc.bad |= SV_BAD_TOKEN;
      if (!valid_uniform(u)) dc.bad |= SV_BAD_U_ACCEPT;
    }
    // A temperature so small that the row maximum over T (log2 units)
    // reaches 2^24 leaves no binary32 room for the exponents of p:
    // invalid data, like a non-finite normaliser.
    if (greedy) s = 1.f;
    else if (!(isfinite(m) && isfinite(s) && fabsf(offset(m, cs)) < kExpLimit))
      dc.bad |= SV_BAD_NORMALISER;
    if (dg.row_max) dg.row_max[static_cast<size_t>(b) * R + i] = m;
    // The normaliser as defined, sum exp2((l - m) * cs): the stored sum
    // times exp2(offset(m) - m * cs), whose exponent one fma forms exactly.
    if (dg.row_sum)
      dg.row_sum[static_cast<size_t>(b) * R + i] =
          greedy ? s : __fmul_rn(s, ex2(-__fmaf_rn(m, cs, -offset(m, cs))));
    if (dg.row_argmax) dg.row_argmax[static_cast<size_t>(b) * R + i] = am;

    if (draft) {
      // Accept test for draft position i.
      const float P = greedy ? ((xc == am) ? 1.f : 0.f)
                             : ex2(__fmaf_rn(lx, cs, -offset(m, cs))) / s;
      const float a = fminf(1.f, P / fmaxf(qraw, kQFloor));
      f = u < a;
      if (dg.p_tok) dg.p_tok[pi] = P;
      if (dg.q_tok) dg.q_tok[pi] = qraw;
      if (dg.accept_prob) dg.accept_prob[pi] = a;
      if (dg.flags) dg.flags[pi] = f ? 1 : 0;
    }
  }
  const unsigned rej = __ballot_sync(kFull, draft && !f);
  if (dc.k < 0 && rej) {
    const int src = __ffs(rej) - 1;
    dc.k = i0 + src;
    dc.mk = __shfl_sync(kFull, m, src);
    dc.sk = __shfl_sync(kFull, s, src);
    dc.ak = __shfl_sync(kFull, am, src);
    dc.xk = __shfl_sync(kFull, x, src);
  }
  if (g >= i0 && g < i0 + 32) {
    dc.mg = __shfl_sync(kFull, m, g - i0);
    dc.sg = __shfl_sync(kFull, s, g - i0);
    dc.ag = __shfl_sync(kFull, am, g - i0);
  }
}

// Warp-wide, after the last group: the request-level checks.  A request
// with invalid data gets -1 tokens and num_accepted, NaN / flag 2
// diagnostics and its error bits (returns false); otherwise the first
// rejection is final, the bonus row if every draft was kept.  Writes
// nothing if out is false.
__device__ __forceinline__ bool close_request(const Params &p, uint32_t *err, int b, int nr,
                                              float t, float us, int lane, Decision &dc,
                                              bool out = true) {
  const int g = nr - 1;
  const int R = p.gmax + 1;
  const sv_diag dg = out ? p.diag : sv_diag{};
  const float qnan = __int_as_float(0x7fc00000);
  if (!valid_temperature(t)) dc.bad |= SV_BAD_TEMPERATURE;
  if (!valid_uniform(us)) dc.bad |= SV_BAD_U_SAMPLE;
  // Diagnostic slots past the request's draft length.
  for (int i = g + lane; i < p.gmax; i += 32) {
    const size_t pi = static_cast<size_t>(b) * p.gmax + i;
    if (dg.p_tok) dg.p_tok[pi] = qnan;
    if (dg.q_tok) dg.q_tok[pi] = qnan;
    if (dg.accept_prob) dg.accept_prob[pi] = qnan;
    if (dg.flags) dg.flags[pi] = 2;
  }
  for (int i = nr + lane; i < R; i += 32) {
    const size_t ri = static_cast<size_t>(b) * R + i;
    if (dg.row_max) dg.row_max[ri] = qnan;
    if (dg.row_sum) dg.row_sum[ri] = qnan;
    if (dg.row_argmax) dg.row_argmax[ri] = -1;
  }
  if (dg.resid_mass && lane == 0) dg.resid_mass[b] = qnan;

  int32_t *tok = p.out_tokens + static_cast<size_t>(b) * R;
  const uint32_t bad = __reduce_or_sync(kFull, dc.bad);
  dc.bad = bad;
  if (bad) {
    if (!out) return false;
    for (int i = lane; i < R; i += 32) tok[i] = -1;
    for (int i = lane; i < p.gmax; i += 32) {
      const size_t pi = static_cast<size_t>(b) * p.gmax + i;
      if (dg.p_tok) dg.p_tok[pi] = qnan;
      if (dg.q_tok) dg.q_tok[pi] = qnan;
      if (dg.accept_prob) dg.accept_prob[pi] = qnan;
      if (dg.flags) dg.flags[pi] = 2;
    }
    for (int i = lane; i < R; i += 32) {
      const size_t ri = static_cast<size_t>(b) * R + i;
      if (dg.row_max) dg.row_max[ri] = qnan;
      if (dg.row_sum) dg.row_sum[ri] = qnan;
      if (dg.row_argmax) dg.row_argmax[ri] = -1;
    }
    if (lane == 0) {
      p.out_nacc[b] = -1;
      atomicOr(err, bad);
      if (dg.accept_hist) atomicAdd(dg.accept_hist + p.gmax + 1, 1);
    }
    return false;
  }
  if (dc.k < 0) {  // every draft kept: the bonus row (tutorial page, §5.3)
    dc.k = g;
    dc.mk = dc.mg;
    dc.sk = dc.sg;
    dc.ak = dc.ag;
    dc.xk = -1;
  }
  return true;
}

// Warp-wide: the accepted drafts, the greedy token at position k, -1 after
// it, num_accepted and the histogram.  A sampled request's position k is
// left to its draw.
__device__ __forceinline__ void write_request(const Params &p, int b, bool greedy, int lane,
                                              const Decision &dc) {
  const int R = p.gmax + 1;
  int32_t *tok = p.out_tokens + static_cast<size_t>(b) * R;
  for (int i = lane; i < R; i += 32) {
    if (i == dc.k && !greedy) continue;
    int tk = -1;
    if (i < dc.k) tk = (i < 32) ? dc.x0 : __ldg(p.ids + static_cast<size_t>(b) * p.gmax + i);
    else if (i == dc.k) tk = dc.ak;
    tok[i] = tk;
  }
  if (lane == 0) {
    p.out_nacc[b] = dc.k;
    if (p.diag.accept_hist) atomicAdd(p.diag.accept_hist + dc.k, 1);
  }
}

// The merge + accept step of request b (nr rows), run by one warp once every
// chunk of its rows is reduced: lane i handles row i.  Its global loads come
// in two waves only: every input that is known up front (request scalars,
// draft ids and uniforms -- or these and the gathers, when the job warp
// fetched them while it waited -- and the first kMergeBatch chunk
// statistics of each row), then the two gathers that need the draft id
// (l_x and q(x)).
template <typename T>
__device__ __noinline__ void merge_request(const Params &p, const Ctl c, int b, int nr, float cs,
                                          int lane, bool pre, DraftIn pin) {
  const int g = nr - 1;
  const int R = p.gmax + 1;
  const bool greedy = (cs == 0.f);

  // A sampled request reserves its descriptor slot first, so the round trip
  // overlaps the loads below; a slot left unused is flagged kReadySkip.
  uint32_t pos = 0;
  if (!greedy && lane == 0) pos = atomicAdd(&c.ctr->b_reserved, 1u);
  // Request-level inputs (the tutorial page, §5.2, takes valid inputs for
  // granted; invalid ones mark only this request).
  const float t = __ldg(p.temp + b);
  const float us = __ldg(p.u_smp + b);

  Decision dc;
  for (int i0 = 0; i0 < nr; i0 += 32) {
    const int i = i0 + lane;
    const bool row = i < nr;
    const Part *pp = p.part1 + (static_cast<size_t>(b) * R + (row ? i : 0)) * p.C1;
    Part q[kMergeBatch];
#pragma unroll
    for (int tj = 0; tj < kMergeBatch; ++tj)
      q[tj] = (row && tj < p.C1) ? ld_cg(pp + tj) : Part{-INFINITY, 0.f};
    const DraftIn in = (pre && i0 == 0) ? pin : load_draft_inputs<T>(p, b, g, greedy, i);
    float m = -INFINITY, s = 0.f;
    int am = -1;
    if (row) {
      // Merge of the chunk statistics, a batch at a time (one batch covers a
      // bf16 row of up to 196608 entries; longer rows take more).  Sums are
      // kept relative to offset(m).
      for (int c0 = 0; c0 < p.C1; c0 += kMergeBatch) {
        if (c0 > 0) {
#pragma unroll
          for (int tj = 0; tj < kMergeBatch; ++tj)
            q[tj] = (c0 + tj < p.C1) ? ld_cg(pp + c0 + tj) : Part{-INFINITY, 0.f};
        }
        fold_batch(q, p.C1 - c0, cs, m, s, am);
      }
    }
    accept_group(p, b, nr, cs, i0, lane, m, s, am, in, dc);
  }
  if (!close_request(p, c.err, b, nr, t, us, lane, dc)) {
    if (lane == 0) {
      if (!greedy) {  // the reserved slot holds nothing: no residual, no search
        p.jflag[p.B + pos] = c.tag | kJobNone;
        c.k2[pos] = kSkipCount;
        desc_publish(p.desc + static_cast<size_t>(pos) * kDescWords, Desc{}, c.tag | kReadySkip);
      }
      count_merged(p, c);
    }
    return;
  }
  if (lane == 0 && !greedy) {
    // Publish first: the slot's residual chunks become claimable once its
    // words are seen (no fence: each word carries the state).
    Desc d;
    d.b = b;
    d.k = dc.k;
    d.slot = b * R + dc.k;
    d.tok = dc.xk;
    d.m = dc.mk;
    d.inv_s = 1.f / dc.sk;
    d.cs = cs;
    d.u = us;
    desc_publish(p.desc + static_cast<size_t>(pos) * kDescWords, d, c.tag | kReadySample);
  }
  write_request(p, b, greedy, lane, dc);
  if (lane == 0) count_merged(p, c);
}

}  // namespace sv
