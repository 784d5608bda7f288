// sv_kv.cuh -- KV rollback hand-off after verification.
//
// Tutorial page dpshk.com/news/5598276 (HTML title 企业官网建设流程全解析),
// §5.4: the KV of the drafted tokens is written first and marked tentative;
// after verification the cache is cut at num_accepted and the blocks past
// the cut go back to the block pool (the corrected token's KV is computed by
// the next step).  For a paged KV cache, per request b with L committed
// tokens, g drafts and k accepted (k < 0: an invalid request, nothing kept):
// blocks [ceil((L + k) / bs), ceil((L + g) / bs)) of block_tables[b] are
// appended to the free list and set to -1, and seq_lens[b] becomes L + k.
#pragma once

#include <cstdint>

#include "spec_verify.h"
#include "sv_device.cuh"

namespace sv {

struct KvParams {
  const int32_t *num_accepted;
  const int32_t *draft_lens;  // NULL: every request has gamma_max drafts
  int32_t *seq_lens;
  int32_t *block_tables;      // [B, max_blocks], -1 = no block
  int B, gamma_max, max_blocks, block_size;
  int32_t *free_list;         // [free_capacity]
  int32_t *free_count;        // device scalar: entries in use
  int free_capacity;
  uint32_t *status;           // SV_KV_* bits, may be NULL
};

constexpr int kKvThreads = 256;

__device__ __forceinline__ int warp_inclusive_scan_int(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// One thread per request; the blocks a warp frees are reserved in the free
// list with one atomicAdd.  Slots at or past the capacity are not written:
// their blocks stay in the table (SV_KV_FREE_LIST_FULL) and the count is
// brought back to the capacity, so that every later reservation starts past
// it and no two writers share a slot.
__global__ void __launch_bounds__(kKvThreads) sv_kv_rollback_kernel(KvParams kp) {
  const int b = blockIdx.x * kKvThreads + threadIdx.x;
  const int lane = threadIdx.x & 31;
  uint32_t st = 0;
  bool valid = false;
  int L = 0, k = 0, kept = 0, used = 0;
  if (b < kp.B) {
    const int g = kp.draft_lens ? kp.draft_lens[b] : kp.gamma_max;
    L = kp.seq_lens[b];
    if (g < 0 || g > kp.gamma_max || L < 0) {
      st |= SV_KV_BAD_LENGTH;
    } else {
      valid = true;
      k = min(max(kp.num_accepted[b], 0), g);
      used = (L + g + kp.block_size - 1) / kp.block_size;
      kept = (L + k + kp.block_size - 1) / kp.block_size;
      if (used > kp.max_blocks) {
        st |= SV_KV_TABLE_SHORT;
        used = kp.max_blocks;
      }
    }
  }
  int32_t *row = kp.block_tables + static_cast<size_t>(valid ? b : 0) * kp.max_blocks;
  int n = 0;
  if (valid) {
    for (int j = kept; j < used; ++j) {
      if (row[j] >= 0) ++n;
      else st |= SV_KV_MISSING_BLOCK;
    }
  }
  const int incl = warp_inclusive_scan_int(n, lane);
  const int tot = __shfl_sync(kFull, incl, 31);
  int base = 0;
  if (lane == 0 && tot) base = atomicAdd(kp.free_count, tot);
  base = __shfl_sync(kFull, base, 0);
  if (valid) {
    int pos = base + incl - n;
    for (int j = kept; j < used; ++j) {
      const int32_t id = row[j];
      if (id < 0) continue;
      if (pos < kp.free_capacity) {
        kp.free_list[pos] = id;
        row[j] = -1;
      } else {
        st |= SV_KV_FREE_LIST_FULL;
      }
      ++pos;
    }
    kp.seq_lens[b] = L + k;
  }
  if (lane == 0 && tot && base + tot > kp.free_capacity) atomicMin(kp.free_count, kp.free_capacity);
  if (st && kp.status) atomicOr(kp.status, st);
}

}  // namespace sv
