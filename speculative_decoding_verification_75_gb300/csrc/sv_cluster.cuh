// sv_cluster.cuh -- the small-batch path: one thread-block cluster per
// request, its CTAs splitting the vocabulary.
//
// Tutorial page dpshk.com/news/5598276 (HTML title 企业官网建设流程全解析),
// §5.2 steps (1)-(5) and §5.3, for batches too small to fill the GPU with
// the persistent kernel's work items.  There the step is a chain of
// dependent latencies (merge, residual, search: each a global round trip or
// several); here every hand-off goes through distributed shared memory:
//
//   1. CTA r of the cluster loads its slice [r W, r W + W) of every row of
//      its request with 1-D TMA copies (all rows at once) and reduces each
//      row slice to (maximum, sum) -- or (maximum, lowest argmax) for a
//      greedy row -- with the same chunk statistics as the persistent kernel;
//   2. each CTA stores its slices' statistics into the shared memory of
//      every CTA of the cluster (distributed shared memory); after a
//      cluster barrier every CTA combines them in rank order from its own
//      shared memory and runs the same accept step (so every CTA knows the
//      first rejection k; only rank 0 writes outputs);
//   3. a sampled request's CTAs form r = (p_k - q_k)_+ (or p_k) on the row-k
//      slice they still hold, loading only their slice of q_k, and sum it per
//      lane run, per warp and per slice;
//   4. the slice sums are pushed the same way; after a second barrier the
//      slice that holds u * S walks its warps, then its lanes' runs, to the
//      token.  No CTA touches a peer's shared memory after that barrier.
//
// The logits are read once (row k is not re-read) and q only at the
// rejected row.  Decisions use the same arithmetic as the persistent path;
// only the grouping of the sums differs (slices of W instead of chunks).
#pragma once

#include "sv_device.cuh"
#include "sv_layout.cuh"
#include "sv_resample.cuh"
#include "sv_rowstats.cuh"

namespace sv {

constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;
constexpr int kCMaxRows = 16;     // gamma_max + 1 at most, for this path
constexpr int kCMaxCluster = 16;  // CTAs per cluster at most

// Elements per warp range of a slice of ne elements: a multiple of 256, so
// that each lane's run (a 32nd of the range) is a whole number of 8-element
// vectors.
__host__ __device__ inline int cluster_warp_range(int ne) {
  const int per = (ne + kCWarps - 1) / kCWarps;
  return (per + 255) / 256 * 256;
}

// Dynamic shared memory of the cluster kernel: one slot of W elements per
// row.  The slice of q_k (fp32: 4 / esz slots) reuses slots of rows other
// than k once the row statistics are done; with fewer than 2 * (4 / esz) + 1
// rows such a run of slots may not exist, and 4 / esz extra slots follow.
__host__ __device__ inline int cluster_q_slots(int esz) { return 4 / esz; }
__host__ __device__ inline int cluster_slots(int rows, int esz) {
  const int ns = cluster_q_slots(esz);
  return rows >= 2 * ns + 1 ? rows : rows + ns;
}
__host__ __device__ inline size_t cluster_smem_bytes(int rows, int W, int esz) {
  return static_cast<size_t>(cluster_slots(rows, esz)) * W * esz;
}
// First slot of q_k's slice: ns slots that do not hold row k.
__host__ __device__ inline int cluster_q_slot(int k, int rows, int esz) {
  const int ns = cluster_q_slots(esz);
  if (k >= ns) return 0;
  return k + 1 + ns <= rows ? k + 1 : rows;
}

template <typename T>
__global__ void __launch_bounds__(kCThreads, 1) sv_cluster_kernel(Params p, int W) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t row_bar_s[kCMaxRows];
  __shared__ uint64_t q_bar_s;
  __shared__ Part wstat_s[kCMaxRows][kCWarps];  // per row, per warp range
  __shared__ float2 part_s[kCMaxCluster][kCMaxRows];  // per rank, per row: slice statistics
  __shared__ float2 wsum_s[kCWarps];            // residual / p sums per warp range
  __shared__ float2 lsum_s[kCWarps][32];        // ... and per lane run
  __shared__ float2 rsum_s[kCMaxCluster];       // ... and of every rank's slice
  __shared__ DraftIn din_s[kCMaxRows];
  __shared__ Ctl ctl_s;
  __shared__ Decision dec_s;
  __shared__ int valid_s;
  __shared__ uint32_t err_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t CS = cluster_size(), rank = cluster_rank();
  const int b = static_cast<int>(blockIdx.x / CS);
  const int R = p.gmax + 1;
  const int e0 = static_cast<int>(rank) * W;
  const int ne = max(0, min(p.V, e0 + W) - e0);
  const int wr = cluster_warp_range(ne);
  const int run = wr / 32;  // elements per lane run
  T *rows = reinterpret_cast<T *>(smem);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kCMaxRows; ++i) mbar_init(smem_addr(&row_bar_s[i]), 1);
    mbar_init(smem_addr(&q_bar_s), 1);
    err_s = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  // Every CTA of the cluster must have started before any writes into a
  // peer's shared memory: arrive now, wait before the first such write.
  cluster_arrive_relaxed();
  pdl_wait();
  pdl_launch_dependents();

  const int nr = request_rows(p, b);
  const int g = nr - 1;
  const float t = __ldg(p.temp + b);
  const float cs = (t > 0.f) ? kLog2e / t : 0.f;
  const bool greedy = cs == 0.f;
  if (threadIdx.x == 0) {  // every row slice of the request, at once
    const uint64_t pol = policy_evict_first();
    for (int i = 0; i < nr; ++i) {
      const uint32_t bar = smem_addr(&row_bar_s[i]);
      if (ne > 0) {
        const uint32_t bytes = static_cast<uint32_t>(ne) * sizeof(T);
        mbar_arrive_expect_tx(bar, bytes);
        tma_load_1d(smem_addr(rows + static_cast<size_t>(i) * W),
                    static_cast<const T *>(p.logits) + (static_cast<size_t>(b) * R + i) * p.V + e0,
                    bytes, bar, pol);
      } else {
        mbar_arrive(bar);
      }
    }
  }
  if (warp == 1 && lane < g) din_s[lane] = load_draft_inputs<T>(p, b, g, greedy, lane);
  if (warp == kCWarps - 1) {
    uint64_t hdr0 = 0, rdy0 = 0, rdy1 = 0;
    if (lane == 0) read_header(p, hdr0, rdy0, rdy1);
    const Ctl c = check_workspace(p, hdr0, rdy0, rdy1, lane, &err_s);
    if (lane == 0) ctl_s = c;
  }

  // 1. Row statistics of this slice, warp range by warp range.
  for (int i = 0; i < nr; ++i) {
    if (!__all_sync(kFull, mbar_wait(smem_addr(&row_bar_s[i]), 0u, &err_s))) break;
    const int off = warp * wr, len = max(0, min(ne, off + wr) - off);
    ChunkStat st = chunk_stats_smem(rows + static_cast<size_t>(i) * W + off, len, cs, lane);
    if (greedy && __float_as_int(st.v) != 0x7fffffff)
      st.v = __int_as_float(__float_as_int(st.v) + e0 + off);  // row index
    if (lane == 0) wstat_s[i][warp] = Part{st.m, st.v};
  }
  __syncthreads();
  cluster_wait();
  if (warp == 0 && lane < nr) {
    Part q[kMergeBatch];
#pragma unroll
    for (int tj = 0; tj < kMergeBatch; ++tj)
      q[tj] = tj < kCWarps ? wstat_s[lane][tj] : Part{-INFINITY, 0.f};
    float m = -INFINITY, s = 0.f;
    int am = -1;
    fold_batch(q, kCWarps, cs, m, s, am);
    // pushed into every CTA of the cluster (this one included): after the
    // barrier each reads them from its own shared memory
    const float2 v = make_float2(m, greedy ? __int_as_float(am) : s);
    for (uint32_t r2 = 0; r2 < CS; ++r2) st_peer_f2(&part_s[rank][lane], r2, v);
  }
  cluster_sync();  // every slice's statistics are in every CTA

  // 2. Every CTA: the rows' statistics over all slices, in rank order, and
  // the accept step; rank 0 writes the outputs.
  const bool out = rank == 0;
  const float us = __ldg(p.u_smp + b);
  if (warp == 0) {
    const Ctl c = ctl_s;
    Decision dc;
    int valid = 0;
    if (nr == 0) {
      if (out && lane == 0) fill_bad_request(p, c, b);
    } else {
      float m = -INFINITY, s = 0.f;
      int am = -1;
      if (lane < nr) {
        Part q[kMergeBatch];
#pragma unroll
        for (int tj = 0; tj < kMergeBatch; ++tj) {
          const float2 v = tj < static_cast<int>(CS) ? part_s[tj][lane]
                                                     : make_float2(-INFINITY, 0.f);
          q[tj] = Part{v.x, v.y};
        }
        fold_batch(q, static_cast<int>(CS), cs, m, s, am);
      }
      const DraftIn in = lane < g ? din_s[lane] : DraftIn{0, 0.f, 0.f, 1.f};
      accept_group(p, b, nr, cs, 0, lane, m, s, am, in, dc, out);
      valid = close_request(p, c.err, b, nr, t, us, lane, dc, out) ? 1 : 0;
      // Accepted drafts, num_accepted; the greedy token (a sampled token
      // is written by the CTA whose slice holds it).
      if (valid && out) write_request(p, b, greedy, lane, dc);
    }
    if (lane == 0) {
      dec_s = dc;
      valid_s = valid;
    }
  }
  __syncthreads();
  const Decision dc = dec_s;

  // 3. A sampled request: r = (p_k - q_k)_+ on this slice (p_k itself for
  // the bonus row), summed per lane run, per warp range and per slice.
  const bool sample = valid_s && !greedy;
  const bool has_q = sample && dc.xk >= 0 && p.q != nullptr;
  // q_k's slice goes to slots no longer needed (every row's statistics are
  // done; row k stays).
  float *qs = reinterpret_cast<float *>(
      rows + static_cast<size_t>(cluster_q_slot(sample ? dc.k : 0, R, sizeof(T))) * W);
  if (has_q && threadIdx.x == 0) {
    // The slots were last read through the generic proxy (the row pass,
    // ordered before this by the barriers above); the copy writes them
    // through the async proxy.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bar = smem_addr(&q_bar_s);
    if (ne > 0) {
      const uint32_t bytes = static_cast<uint32_t>(ne) * 4u;
      mbar_arrive_expect_tx(bar, bytes);
      tma_load_1d(smem_addr(qs), p.q + (static_cast<size_t>(b) * p.gmax + dc.k) * p.V + e0,
                  bytes, bar, policy_evict_first());
    } else {
      mbar_arrive(bar);
    }
  }
  const T *xk_row = rows + static_cast<size_t>(dc.k) * W;
  const float nego = -__fmul_rn(dc.mk, cs), inv_s = 1.f / dc.sk;
  // p_j and r_j of eight consecutive slice elements j0 .. j0+7 (j0 a
  // multiple of 8; runs are whole 8-element vectors, and elements past the
  // slice end -- an fp32 slice may end 4 elements into a vector -- weigh
  // nothing).  Computed together so that the loads and exponentials of the
  // eight overlap; the sums below still add them one after another, in
  // order.  At a deterministic draft's token the residual is 0 exactly
  // (q = 1 there, and p <= 1 up to rounding).
  auto weights8 = [&](int j0, float (&pw)[8], float (&rw)[8]) {
    float x[8], qv[8];
    if constexpr (sizeof(T) == 2) {
      const uint4 w = *reinterpret_cast<const uint4 *>(xk_row + j0);
      x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
      x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
    } else {
      const float4 a = *reinterpret_cast<const float4 *>(xk_row + j0);
      const float4 c4 = *reinterpret_cast<const float4 *>(xk_row + j0 + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = c4.x; x[5] = c4.y; x[6] = c4.z; x[7] = c4.w;
    }
    if (has_q) {
      const float4 a = *reinterpret_cast<const float4 *>(qs + j0);
      const float4 c4 = *reinterpret_cast<const float4 *>(qs + j0 + 4);
      qv[0] = a.x; qv[1] = a.y; qv[2] = a.z; qv[3] = a.w;
      qv[4] = c4.x; qv[5] = c4.y; qv[6] = c4.z; qv[7] = c4.w;
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) qv[u] = (dc.xk >= 0 && e0 + j0 + u == dc.xk) ? 1.f : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = j0 + u < ne;
      pw[u] = in ? target_p(x[u], nego, cs, inv_s) : 0.f;
      rw[u] = in ? resid(pw[u], qv[u]) : 0.f;  // q = 0 on the bonus row: r = p
      if (!has_q && dc.xk >= 0 && e0 + j0 + u == dc.xk) rw[u] = 0.f;
    }
  };
  if (sample) {
    bool ok = true;
    if (has_q) ok = __all_sync(kFull, mbar_wait(smem_addr(&q_bar_s), 0u, &err_s));
    const int l0 = warp * wr + lane * run;
    float lr = 0.f, lp = 0.f;
    if (ok) {
      for (int j0 = l0; j0 < min(l0 + run, ne); j0 += 8) {
        float pw[8], rw[8];
        weights8(j0, pw, rw);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          lr = __fadd_rn(lr, rw[u]);
          lp = __fadd_rn(lp, pw[u]);
        }
      }
    }
    lsum_s[warp][lane] = make_float2(lr, lp);
    const float ir = warp_inclusive_scan(lr, lane), ip = warp_inclusive_scan(lp, lane);
    if (lane == 31) wsum_s[warp] = make_float2(ir, ip);
    __syncthreads();
    if (threadIdx.x == 0) {
      float sr = 0.f, sp = 0.f;
      for (int w = 0; w < kCWarps; ++w) {
        sr = __fadd_rn(sr, wsum_s[w].x);
        sp = __fadd_rn(sp, wsum_s[w].y);
      }
      for (uint32_t r2 = 0; r2 < CS; ++r2) st_peer_f2(&rsum_s[rank], r2, make_float2(sr, sp));
    }
  }
  // Every slice's sums are in every CTA.  No CTA touches a peer's shared
  // memory after this barrier, so each may leave when it is done.
  cluster_sync();

  // 4. The draw: the slice, then the warp range, then the lane run holding
  // u * S (S the residual mass, or p's when the residual is empty).
  __shared__ int draw_warp_s;
  __shared__ float draw_base_s, draw_target_s;
  __shared__ int draw_use_p_s;
  if (sample && warp == 0) {
    const float2 v = lane < static_cast<int>(CS) ? rsum_s[lane] : make_float2(0.f, 0.f);
    const float tr = __shfl_sync(kFull, warp_inclusive_scan(v.x, lane), 31);
    const float tp = __shfl_sync(kFull, warp_inclusive_scan(v.y, lane), 31);
    const bool use_p = !(tr > 0.f);  // empty residual: draw from p itself
    float target = __fmul_rn(us, use_p ? tp : tr);
    bool fb = false;
    float base = 0.f;
    const int rs = max(0, cdf_level64(static_cast<int>(CS), use_p ? v.y : v.x, 0.f, 0.f, target,
                                      lane, &base, &fb));
    if (fb) target = INFINITY;  // rounding pushed u*S past the total
    int ws = -1;
    if (rs == static_cast<int>(rank)) {
      const float ww = lane < kCWarps ? (use_p ? wsum_s[lane].y : wsum_s[lane].x) : 0.f;
      bool fb2 = false;
      float base2 = base;
      ws = max(0, cdf_level64(kCWarps, ww, 0.f, base, target, lane, &base2, &fb2));
      if (fb2) target = INFINITY;
      base = base2;
    }
    if (lane == 0) {
      draw_warp_s = ws;
      draw_base_s = base;
      draw_target_s = target;
      draw_use_p_s = use_p ? 1 : 0;
      if (out && p.diag.resid_mass) p.diag.resid_mass[b] = tr;
    }
  }
  __syncthreads();
  if (sample && warp == draw_warp_s) {
    const bool use_p = draw_use_p_s != 0;
    const float base = draw_base_s, target = draw_target_s;
    const float lw = use_p ? lsum_s[warp][lane].y : lsum_s[warp][lane].x;
    const float incl = base + warp_inclusive_scan(lw, lane);
    const float prev = __shfl_up_sync(kFull, incl, 1);
    const float excl = (lane == 0) ? base : prev;
    int tok = -1;
    // The first lane with weight whose inclusive prefix passes the target
    // holds the token (as at every level of the draw, an index without
    // weight is never chosen, even where rounding puts its prefix past the
    // target).  For runs of more than two vectors the whole warp walks that
    // lane's run, a vector of 8 per lane, each vector from its exclusive
    // prefix within the run: one vector's weights per lane instead of a
    // run's (8 requests at V = 151936: 14.1 vs 14.9 us a step; for shorter
    // runs the extra scan costs more than it saves).
    const unsigned pass = __ballot_sync(kFull, lw > 0.f && incl > target);
    if (pass && run > 16 && run <= 8 * 32) {
      const int L = __ffs(pass) - 1;
      const float start = __shfl_sync(kFull, excl, L);
      const int j0 = warp * wr + L * run + 8 * lane;
      const bool mine = 8 * lane < run && j0 < ne;
      float pw[8], rw[8];
      float vs = 0.f;
      if (mine) {
        weights8(j0, pw, rw);
#pragma unroll
        for (int u = 0; u < 8; ++u) vs = __fadd_rn(vs, use_p ? pw[u] : rw[u]);
      }
      const float vincl = warp_inclusive_scan(vs, lane);
      const float vprev = __shfl_up_sync(kFull, vincl, 1);
      float c = (lane == 0) ? start : __fadd_rn(start, vprev);
      int hit = -1;
      if (mine) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float wu = use_p ? pw[u] : rw[u];
          c = __fadd_rn(c, wu);
          if (hit < 0 && wu > 0.f && c > target) hit = j0 + u;
        }
      }
      const unsigned hb = __ballot_sync(kFull, hit >= 0);
      if (hb) tok = e0 + __shfl_sync(kFull, hit, __ffs(hb) - 1);
    }
    if (tok < 0) {
      // Rounding kept the walk of that run below the target, or u*S lies at
      // or past the total: each lane walks its own run from its exclusive
      // prefix; the first lane to pass the target holds the token, else the
      // last positive weight.
      float c = excl;
      const int l0 = warp * wr + lane * run;
      int hit = -1, lastpos = -1;
      for (int j0 = l0; j0 < min(l0 + run, ne) && hit < 0; j0 += 8) {
        float pw[8], rw[8];
        weights8(j0, pw, rw);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float w = use_p ? pw[u] : rw[u];
          c = __fadd_rn(c, w);
          if (hit < 0 && w > 0.f && c > target) hit = j0 + u;
          if (w > 0.f) lastpos = j0 + u;
        }
      }
      tok = e0;
      const unsigned hb = __ballot_sync(kFull, hit >= 0);
      if (hb) {
        tok = e0 + __shfl_sync(kFull, hit, __ffs(hb) - 1);
      } else {
        const unsigned pb = __ballot_sync(kFull, lastpos >= 0);
        if (pb) tok = e0 + __shfl_sync(kFull, lastpos, 31 - __clz(pb));
      }
    }
    if (lane == 0) p.out_tokens[static_cast<size_t>(b) * R + dc.k] = tok;
  }

  if (threadIdx.x == 0) {
    // The call's error word, and the epoch: the grid's last CTA advances it.
    const Ctl c = ctl_s;
    const uint32_t f = err_s;
    if (f) atomicOr(c.err, f);
    if (f || !c.ok) {
      st_relaxed64(&p.hdr->ready[0], 0ull);
      st_relaxed64(&p.hdr->ready[1], 0ull);
    }
    if (atomicAdd(&c.ctr->exited, 1u) == gridDim.x - 1) st_relaxed(&p.hdr->epoch, c.epoch + 1u);
  }
}

}  // namespace sv
