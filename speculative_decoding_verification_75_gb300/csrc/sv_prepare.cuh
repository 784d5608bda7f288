// sv_prepare.cuh -- kernel 0: reset the workspace's counters for this call.
//
// One CTA clears the per-request arrival counters and the header, and writes
// the -1 outputs of requests whose draft length is invalid (they have no rows
// for the row-statistics kernel to stream).  Every other per-request check
// happens in the row-statistics kernel's merge step.  The row-statistics
// kernel streams logits while this runs; it waits for this grid only before
// its first counter update.
#pragma once

#include "sv_device.cuh"
#include "sv_layout.cuh"

namespace sv {

constexpr int kPrepThreads = 1024;

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
  pdl_launch_dependents();
  __shared__ uint32_t err_acc;
  if (threadIdx.x == 0) err_acc = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < p.B; b += kPrepThreads) {
    p.k1_cnt[b] = 0u;
    p.k2_cnt[b] = 0u;
    if (request_rows(p, b) == 0) {
      fill_bad_request(p, b);
      atomicOr(&err_acc, SV_BAD_DRAFT_LEN);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.hdr->err = err_acc;
    p.hdr->n_q = 0u;
    p.hdr->n_noq = 0u;
    p.hdr->k2_next = 0u;
  }
}

}  // namespace sv
