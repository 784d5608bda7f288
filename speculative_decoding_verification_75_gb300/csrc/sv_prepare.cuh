// sv_prepare.cuh -- kernel 0: per-call tables for batches too large for the
// persistent kernel's shared memory, and the reset of the caller's
// acceptance histogram.
//
// For up to kSmemReq requests every CTA of the persistent kernel builds its
// own copy of the tables in shared memory and this kernel is not launched
// (unless the call asks for the histogram).  Otherwise one CTA walks the
// batch 256 requests at a time: it writes each request's first flat row (an
// exclusive scan of g_b + 1) and softmax scale log2(e)/T.
#pragma once

#include "sv_device.cuh"
#include "sv_layout.cuh"

namespace sv {

// Small enough to sit beside a persistent CTA on one SM (registers, threads),
// so that it can be resident while the previous step's grid finishes.
constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;

__global__ void __launch_bounds__(kPrepThreads) sv_prepare_kernel(Params p) {
  // Launched as a programmatic dependent: it may be resident before the
  // previous grid on the stream has finished, so it waits for that grid's
  // completion (and memory) before touching anything.  The persistent
  // kernel may then start its prologue; it waits for this grid's completion
  // before it reads anything written here.
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int warp_tot[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (p.diag.accept_hist)
    for (int j = tid; j < p.gmax + 2; j += kPrepThreads) p.diag.accept_hist[j] = 0;
  if (!p.tables_global) return;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < p.B; base += kPrepThreads) {
    const int b = base + tid;
    int nr = 0;
    if (b < p.B) {
      nr = request_rows(p, b);
      const float t = __ldg(p.temp + b);
      p.cs[b] = (t > 0.f) ? kLog2e / t : 0.f;
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
  if (tid == 0) p.row_start[p.B] = carry;
}

}  // namespace sv
