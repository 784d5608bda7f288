// sv_rowstats.cuh -- kernel 1: target-softmax statistics of every row, then
// the accept test and first-rejection scan of every request.
//
// Tutorial page dpshk.com/news/5598276 (HTML title 企业官网建设流程全解析),
// §5.2 steps (1)-(4): softmax of the g+1 target rows, a_i = min(1, p/q) with
// q clamped at 1e-10, accepted = u < a, cumprod prefix = first rejection.
//
// Work decomposition.  The vocabulary of every active row is cut into
// 16 KiB chunks (8192 bf16 or 4096 fp32 logits); the flat list of (row,
// chunk) items is split into equal contiguous ranges, one per persistent CTA.
// Each CTA finds where its range starts by a block-wide scan of the draft
// lengths, so streaming does not wait for any other kernel.  One producer
// lane streams the range with 1-D TMA bulk copies into a ring of shared-
// memory stages, and consumer warps each reduce one whole chunk: pass A takes
// the maximum (packed bf16x2 max), pass B the sum of exp2((l - max) *
// log2(e)/T) with packed fp32x2 arithmetic (greedy rows instead find the
// lowest index of the maximum).  p itself is never stored: only (max, sum)
// per chunk reaches global memory.
//
// Completion is counted in two levels: chunks of a request within the CTA on
// a shared-memory counter (CTA-scope release/acquire), then one GPU-scope
// atomic per CTA and request.  The CTA that completes a request (no waiting)
// merges its chunk statistics in chunk order, checks the request's inputs,
// gathers p(x_i) and q(x_i), runs the accept test for all positions with one
// ballot, writes the accepted drafts and queues the row to re-sample for
// kernel 2.
#pragma once

#include "sv_device.cuh"
#include "sv_layout.cuh"

namespace sv {

// Pipeline shape: kK1Stages 16 KiB stages shared by kK1Consumers warps (each
// owns kK1Stages / kK1Consumers of them).  Measured on GB300 at B=128, g=5,
// V=151936: one stage per warp with 12 warps beats two per warp with 6, the
// chunk reductions need the extra warps more than the extra buffering.
#ifndef SV_K1_CONSUMERS
#define SV_K1_CONSUMERS 12
#endif
#ifndef SV_K1_STAGES
#define SV_K1_STAGES 12
#endif
constexpr int kK1Consumers = SV_K1_CONSUMERS;
constexpr int kK1Stages = SV_K1_STAGES;
constexpr int kK1StageBytes = 16384;
constexpr int kK1Threads = 32 * (kK1Consumers + 1);
constexpr int kLocalSlots = 32;   // > kK1Stages: see the slot-reuse note below
static_assert(kK1Stages % kK1Consumers == 0, "each consumer warp owns whole stages");
static_assert(kLocalSlots > kK1Stages, "a local counter slot is reused only after "
                                       "every item of its previous request is counted");

struct ItemInfo {
  int slot;     // padded row index b*(gamma_max+1)+i (-1: end of stream)
  int c;        // chunk within the row
  int ne;       // elements in the chunk
  float cs;     // log2(e) / T (0: greedy)
  int b;        // request
  int lslot;    // shared-memory counter of the request in this CTA
  int ltotal;   // items of the request inside this CTA's range
  int gtotal;   // items of the request overall (rows * chunks)
};

constexpr size_t k1_smem_bytes() {
  return static_cast<size_t>(kK1Stages) * kK1StageBytes +
         kK1Stages * sizeof(ItemInfo) + 2 * kK1Stages * sizeof(uint64_t);
}

__device__ __forceinline__ uint32_t atomic_add_acq_rel_cta(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.cta.shared::cta.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}

// ------------------------------------------------- chunk statistics ----

struct ChunkStat {
  float m;  // maximum logit of the chunk
  float v;  // sum of exp2((l - m) * cs), or the argmax bits for greedy rows
};

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162 *>(&a),
                             *reinterpret_cast<__nv_bfloat162 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// exp2((x - m) * cs) for a pair, packed fp32x2 arithmetic.
__device__ __forceinline__ float2 exp_pair(float2 x, float2 negm, float2 cs2) {
  const float2 t = __fmul2_rn(__fadd2_rn(x, negm), cs2);
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
    const float2 negm = make_float2(-m, -m), cs2 = make_float2(cs, cs);
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll 4
    for (int i = lane; i < nvec; i += 32) {
      const uint4 x = v[i];
      a0 = __fadd2_rn(a0, exp_pair(make_float2(bf16_lo(x.x), bf16_hi(x.x)), negm, cs2));
      a1 = __fadd2_rn(a1, exp_pair(make_float2(bf16_lo(x.y), bf16_hi(x.y)), negm, cs2));
      a0 = __fadd2_rn(a0, exp_pair(make_float2(bf16_lo(x.z), bf16_hi(x.z)), negm, cs2));
      a1 = __fadd2_rn(a1, exp_pair(make_float2(bf16_lo(x.w), bf16_hi(x.w)), negm, cs2));
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
    const float2 negm = make_float2(-m, -m), cs2 = make_float2(cs, cs);
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll 4
    for (int i = lane; i < nvec; i += 32) {
      const float4 x = v[i];
      a0 = __fadd2_rn(a0, exp_pair(make_float2(x.x, x.y), negm, cs2));
      a1 = __fadd2_rn(a1, exp_pair(make_float2(x.z, x.w), negm, cs2));
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
    float s = 0.f;
    for (int j = lane; j < ne; j += 32)
      s += ex2(__fmul_rn(__fsub_rn(Elem<T>::load(row, e0 + j), m), cs));
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

// ----------------------------------------- merge + accept (last arriver) ----

template <typename T>
__device__ void merge_request(const Params &p, int b, int nr, float cs, int lane) {
  const int g = nr - 1;
  const int R = p.gmax + 1;
  const bool greedy = (cs == 0.f);
  const T *logits = static_cast<const T *>(p.logits);
  const sv_diag &dg = p.diag;
  const float qnan = __int_as_float(0x7fc00000);

  // Request-level checks (P3 §5.2 takes valid inputs for granted; invalid
  // ones mark only this request).
  const float t = __ldg(p.temp + b);
  const float us = __ldg(p.u_smp + b);
  uint32_t bad = 0;
  if (!valid_temperature(t)) bad |= SV_BAD_TEMPERATURE;
  if (!valid_uniform(us)) bad |= SV_BAD_U_SAMPLE;

  int k = -1;                       // first rejected position
  float mk = 0.f, sk = 1.f;         // its row statistics
  int ak = -1;
  float mg = 0.f, sg = 1.f;         // bonus row statistics
  int ag = -1;

  for (int i0 = 0; i0 < nr; i0 += 32) {
    const int i = i0 + lane;
    float m = -INFINITY, s = 0.f;
    int am = -1;
    bool f = true;
    if (i < nr) {
      // Draft-position inputs first: their loads overlap the merge below.
      const size_t pi = static_cast<size_t>(b) * p.gmax + i;
      int x = 0;
      float lx = 0.f, qraw = 1.f, u = 0.f;
      if (i < g) {
        x = __ldg(p.ids + pi);
        u = __ldg(p.u_acc + pi);
        if (x < 0 || x >= p.V) {
          bad |= SV_BAD_TOKEN;
          x = 0;
        }
        if (!valid_uniform(u)) bad |= SV_BAD_U_ACCEPT;
        if (!greedy) lx = Elem<T>::load(logits, (static_cast<size_t>(b) * R + i) * p.V + x);
        if (p.q) qraw = __ldg(p.q + pi * p.V + x);
      }
      // Online merge of the chunk statistics in chunk order, loads batched
      // eight at a time so their latencies overlap.
      const Part *pp = p.part1 + (static_cast<size_t>(b) * R + i) * p.C;
      for (int c0 = 0; c0 < p.C; c0 += 8) {
        Part q[8];
#pragma unroll
        for (int t8 = 0; t8 < 8; ++t8)
          q[t8] = (c0 + t8 < p.C) ? ld_cg(pp + c0 + t8) : Part{-INFINITY, 0.f};
#pragma unroll
        for (int t8 = 0; t8 < 8; ++t8) {
          if (c0 + t8 >= p.C) break;
          if (greedy) {
            if (q[t8].m > m || am < 0) {
              m = q[t8].m;
              am = __float_as_int(q[t8].v);
            }
          } else if (q[t8].m > m) {
            s = __fadd_rn(__fmul_rn(s, ex2(__fmul_rn(__fsub_rn(m, q[t8].m), cs))), q[t8].v);
            m = q[t8].m;
          } else if (q[t8].m != -INFINITY) {
            s = __fadd_rn(s, __fmul_rn(q[t8].v, ex2(__fmul_rn(__fsub_rn(q[t8].m, m), cs))));
          }
        }
      }
      if (greedy) s = 1.f;
      else if (!(isfinite(m) && isfinite(s))) bad |= SV_BAD_NORMALISER;
      if (dg.row_max) dg.row_max[static_cast<size_t>(b) * R + i] = m;
      if (dg.row_sum) dg.row_sum[static_cast<size_t>(b) * R + i] = s;
      if (dg.row_argmax) dg.row_argmax[static_cast<size_t>(b) * R + i] = am;

      if (i < g) {
        // Accept test for draft position i.
        const float P = greedy ? ((x == am) ? 1.f : 0.f)
                               : ex2(__fmul_rn(__fsub_rn(lx, m), cs)) / s;
        const float a = fminf(1.f, P / fmaxf(qraw, kQFloor));
        f = u < a;
        if (dg.p_tok) dg.p_tok[pi] = P;
        if (dg.q_tok) dg.q_tok[pi] = qraw;
        if (dg.accept_prob) dg.accept_prob[pi] = a;
        if (dg.flags) dg.flags[pi] = f ? 1 : 0;
      }
    }
    const unsigned rej = __ballot_sync(kFull, i < g && !f);
    if (k < 0 && rej) {
      const int src = __ffs(rej) - 1;
      k = i0 + src;
      mk = __shfl_sync(kFull, m, src);
      sk = __shfl_sync(kFull, s, src);
      ak = __shfl_sync(kFull, am, src);
    }
    if (g >= i0 && g < i0 + 32) {
      mg = __shfl_sync(kFull, m, g - i0);
      sg = __shfl_sync(kFull, s, g - i0);
      ag = __shfl_sync(kFull, am, g - i0);
    }
  }
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
  bad = __reduce_or_sync(kFull, bad);
  if (bad) {
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
      atomicOr(&p.hdr->err, bad);
    }
    return;
  }
  if (k < 0) {  // every draft kept: the bonus row (P3 §5.3)
    k = g;
    mk = mg;
    sk = sg;
    ak = ag;
  }
  for (int i = lane; i < R; i += 32) {
    int tk = -1;
    if (i < k) tk = __ldg(p.ids + static_cast<size_t>(b) * p.gmax + i);
    else if (i == k && greedy) tk = ak;
    tok[i] = tk;
  }
  if (lane == 0) {
    p.out_nacc[b] = k;
    if (!greedy) {
      Desc d;
      d.b = b;
      d.k = k;
      d.slot = b * R + k;
      d.tok = (k < g) ? __ldg(p.ids + static_cast<size_t>(b) * p.gmax + k) : -1;
      d.m = mk;
      d.inv_s = 1.f / sk;
      d.cs = cs;
      d.u = us;
      const bool has_q = (k < g) && p.q != nullptr;
      if (has_q) {
        const uint32_t pos = atomicAdd(&p.hdr->n_q, 1u);
        p.desc_q[pos] = d;
      } else {
        const uint32_t pos = atomicAdd(&p.hdr->n_noq, 1u);
        p.desc_noq[pos] = d;
      }
    }
  }
}

// ------------------------------------------------------------- kernel ----

// Block-wide exclusive scan of one int per thread; also returns the total.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += n;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  const int r = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - v;
  *total = warp_tot[nw - 1];
  return r;
}

template <typename T, bool kTMA>
__global__ void __launch_bounds__(kK1Threads, 1) sv_rowstats_kernel(Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t lcnt[kLocalSlots];
  __shared__ int warp_tot[32];
  __shared__ int s_b0, s_rs0;
  ItemInfo *info = reinterpret_cast<ItemInfo *>(smem + kK1Stages * kK1StageBytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(info + kK1Stages);
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kK1Stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.gmax + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kK1Stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    fence_mbar_init();
  }
  if (threadIdx.x < kLocalSlots) lcnt[threadIdx.x] = 0u;

  // Where does this CTA's range of (row, chunk) items start?  Rows are
  // counted over requests in order; each thread sums a contiguous block.
  const int per = (p.B + kK1Threads - 1) / kK1Threads;
  const int bb = min(p.B, static_cast<int>(threadIdx.x) * per), be = min(p.B, bb + per);
  int my = 0;
  if (p.lens) {
    for (int b = bb; b < be; ++b) my += request_rows(p, b);
  } else {
    my = (be - bb) * R;
  }
  int n_rows = 0;
  const int excl = block_excl_scan(my, warp_tot, &n_rows);
  const long long n_items = static_cast<long long>(n_rows) * p.C;
  const long long lo = n_items * blockIdx.x / gridDim.x;
  const long long hi = n_items * (blockIdx.x + 1) / gridDim.x;
  if (lo < hi) {
    const long long fr_lo = lo / p.C;
    if (excl <= fr_lo && fr_lo < excl + my) {
      int acc = excl;
      for (int b = bb; b < be; ++b) {
        const int nr = request_rows(p, b);
        if (fr_lo < acc + nr) {
          s_b0 = b;
          s_rs0 = acc;
          break;
        }
        acc += nr;
      }
    }
  }
  __syncthreads();
  pdl_launch_dependents();

  const T *logits = static_cast<const T *>(p.logits);
  constexpr int kChunk = Elem<T>::kChunk;
  static_assert(kChunk * sizeof(T) == kK1StageBytes, "one chunk per stage");
  uint32_t *err = &p.hdr->err;

  if (warp == 0) {
    if (lane != 0) return;
    // ------------------------------------------------ producer lane ----
    const uint64_t pol = policy_evict_normal();
    uint32_t n = 0;
    bool ok = true;
    if (lo < hi) {
      int b = s_b0, rs = s_rs0, j = 0;
      int nr = request_rows(p, b);
      float cs = 0.f;
      int ltotal = 0, gtotal = 0;
      bool fresh = true;
      // (row, chunk) advanced incrementally: this lane issues every copy of
      // the CTA, and a 64-bit division per item would make it the bottleneck.
      int fr = static_cast<int>(lo / p.C), c = static_cast<int>(lo - static_cast<long long>(fr) * p.C);
      for (long long it = lo; it < hi; ++it, ++n, (++c == p.C ? (c = 0, ++fr) : 0)) {
        while (fr >= rs + nr) {  // next request with rows
          rs += nr;
          ++b;
          nr = request_rows(p, b);
          fresh = true;
        }
        if (fresh) {
          const float t = __ldg(p.temp + b);
          cs = (t > 0.f) ? kLog2e / t : 0.f;
          gtotal = nr * p.C;
          const long long rlo = static_cast<long long>(rs) * p.C;
          const long long rhi = static_cast<long long>(rs + nr) * p.C;
          ltotal = static_cast<int>(min(hi, rhi) - max(lo, rlo));
          if (it != lo) ++j;
          fresh = false;
        }
        const int slot = b * R + (fr - rs);
        const int e0 = c * kChunk, ne = min(kChunk, p.V - e0);
        const int s = static_cast<int>(n % kK1Stages);
        const uint32_t ph = (n / kK1Stages) & 1u;
        if (n >= kK1Stages && !(ok = mbar_wait(empty0 + 8 * s, ph ^ 1u, err))) break;
        info[s] = ItemInfo{slot, c, ne, cs, b, j % kLocalSlots, ltotal, gtotal};
        if (kTMA) {
          const uint32_t bytes = static_cast<uint32_t>(ne) * sizeof(T);
          mbar_arrive_expect_tx(full0 + 8 * s, bytes);
          tma_load_1d(smem_addr(smem + static_cast<size_t>(s) * kK1StageBytes),
                      logits + static_cast<size_t>(slot) * p.V + e0, bytes, full0 + 8 * s, pol);
        } else {
          mbar_arrive(full0 + 8 * s);
        }
      }
    }
    // One end-of-stream marker per consumer warp.
    for (int w = 0; ok && w < kK1Consumers; ++w, ++n) {
      const int s = static_cast<int>(n % kK1Stages);
      const uint32_t ph = static_cast<uint32_t>((n / kK1Stages) & 1);
      if (n >= kK1Stages && !(ok = mbar_wait(empty0 + 8 * s, ph ^ 1u, err))) break;
      info[s].slot = -1;
      mbar_arrive(full0 + 8 * s);
    }
    // Every copy this CTA issued must have landed before it exits.
    for (uint32_t jj = (n > kK1Stages ? n - kK1Stages : 0); jj < n; ++jj)
      mbar_wait(full0 + 8 * static_cast<int>(jj % kK1Stages),
                static_cast<uint32_t>((jj / kK1Stages) & 1), err);
    return;
  }

  // ---------------------------------------------------- consumer warps ----
  // Local slot reuse: an item is released (empty barrier) only after it was
  // counted, and the producer issues item n only after item n - kK1Stages was
  // released; a request's slot comes back kLocalSlots > kK1Stages requests
  // later, so all of the previous owner's items are counted by then.
  const int cw = warp - 1;
  bool waited = false;
  for (uint32_t n = cw;; n += kK1Consumers) {
    const int s = static_cast<int>(n % kK1Stages);
    const uint32_t ph = static_cast<uint32_t>((n / kK1Stages) & 1);
    if (!mbar_wait(full0 + 8 * s, ph, err)) break;
    const ItemInfo inf = info[s];
    if (inf.slot < 0) break;
    ChunkStat st;
    if (kTMA) {
      st = chunk_stats_smem(
          reinterpret_cast<const T *>(smem + static_cast<size_t>(s) * kK1StageBytes),
          inf.ne, inf.cs, lane);
    } else {
      st = chunk_stats_global<T>(logits + static_cast<size_t>(inf.slot) * p.V,
                                 inf.c * kChunk, inf.ne, inf.cs, lane);
    }
    if (inf.cs == 0.f && __float_as_int(st.v) != 0x7fffffff)
      st.v = __int_as_float(__float_as_int(st.v) + inf.c * kChunk);
    if (!waited) {
      pdl_wait();  // the counters were reset by kernel 0
      waited = true;
    }
    int last = 0;
    if (lane == 0) {
      p.part1[static_cast<size_t>(inf.slot) * p.C + inf.c] = Part{st.m, st.v};
      if (atomic_add_acq_rel_cta(&lcnt[inf.lslot], 1u) + 1 == static_cast<uint32_t>(inf.ltotal)) {
        lcnt[inf.lslot] = 0u;
        const uint32_t old = atomic_add_acq_rel(&p.k1_cnt[inf.b], static_cast<uint32_t>(inf.ltotal));
        last = (old + inf.ltotal == static_cast<uint32_t>(inf.gtotal));
      }
      mbar_arrive(empty0 + 8 * s);
    }
    if (__shfl_sync(kFull, last, 0)) {
      __threadfence();
      merge_request<T>(p, inf.b, inf.gtotal / p.C, inf.cs, lane);
    }
  }
}

}  // namespace sv
