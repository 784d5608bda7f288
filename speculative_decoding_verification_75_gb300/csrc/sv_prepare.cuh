// sv_prepare.cuh -- kernel 0: per-call set-up of the workspace.
//
// One CTA walks the batch 256 requests at a time: it writes each request's
// first flat row (an exclusive scan of g_b + 1) and softmax scale log2(e)/T,
// clears the request's arrival counters and descriptor flag, and writes the
// -1 outputs of requests whose draft length is invalid (they get no rows).
// Every other per-request check happens in the merge step.  It also resets
// the header: error word, row and request totals, and the work counters of
// the persistent kernel.
#pragma once

#include "sv_device.cuh"
#include "sv_layout.cuh"

namespace sv {

// Small enough to sit beside a persistent CTA on one SM (registers, threads),
// so that it can be resident while the previous step's grid finishes.
constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;

__device__ void fill_bad_request(const Params &p, int b) {
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
}

__global__ void __launch_bounds__(kPrepThreads) sv_prepare_kernel(Params p) {
  // Launched as a programmatic dependent: it may be resident before the
  // previous grid on the stream has finished, so it waits for that grid's
  // completion (and memory) before touching anything.  The persistent
  // kernel may then start its prologue; it waits for this grid's completion
  // before it reads anything written here.
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int warp_tot[32];
  __shared__ int carry, valid;
  __shared__ uint32_t err_acc;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (p.diag.accept_hist)
    for (int j = tid; j < p.gmax + 2; j += kPrepThreads) p.diag.accept_hist[j] = 0;
  if (tid == 0) {
    carry = 0;
    valid = 0;
    err_acc = 0;
  }
  __syncthreads();
  for (int base = 0; base < p.B; base += kPrepThreads) {
    const int b = base + tid;
    int nr = 0;
    if (b < p.B) {
      nr = request_rows(p, b);
      const float t = __ldg(p.temp + b);
      p.cs[b] = (t > 0.f) ? kLog2e / t : 0.f;
      p.k1_cnt[b] = 0u;
      p.k2_cnt[b] = 0u;
      for (int i = 0; i < kDescWords; ++i) p.desc[static_cast<size_t>(b) * kDescWords + i] = 0ull;
      p.jflag[b] = nr == 0 ? kJobNone : kJobWait;  // no merge without rows
      p.jflag[p.B + b] = kJobWait;
      if (nr == 0) {
        fill_bad_request(p, b);
        atomicOr(&err_acc, SV_BAD_DRAFT_LEN);
        if (p.diag.accept_hist) atomicAdd(p.diag.accept_hist + p.gmax + 1, 1);
      } else {
        atomicAdd(&valid, 1);
      }
    }
    // Exclusive scan of the row counts: first flat row of each request.
    int incl = nr;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kPrepWarps ? warp_tot[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, w, o);
        if (lane >= o) w += n;
      }
      warp_tot[lane] = w;
    }
    __syncthreads();
    if (b < p.B) p.row_start[b] = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - nr;
    __syncthreads();
    if (tid == 0) carry += warp_tot[kPrepWarps - 1];
    __syncthreads();
  }
  if (tid == 0) {
    p.row_start[p.B] = carry;
    p.hdr->err = err_acc;
    p.hdr->n_rows = static_cast<uint32_t>(carry);
    p.hdr->n_valid = static_cast<uint32_t>(valid);
    p.hdr->a_next = 0u;
    p.hdr->b_next = 0u;
    p.hdr->b_reserved = 0u;
    p.hdr->n_merged = 0u;
    p.hdr->jq_head = 0u;
    p.hdr->all_merged = valid == 0 ? 1u : 0u;  // nothing to merge
  }
}

}  // namespace sv
