// sv_verify.cuh -- the persistent verification kernel.
//
// One CTA per SM runs the whole verification step of a batch in one launch
// (the small set-up kernel 0 runs first only for batches beyond the shared
// tables' 256 requests or when the acceptance histogram is asked for), on
// two kinds of work item:
//
//   row-statistics items  every (active row, vocabulary chunk) of the target
//                         logits, handed out from a global counter in blocks,
//                         request after request (tutorial page
//                         dpshk.com/news/5598276, §5.2 steps (1)-(4));
//   residual items        for each request that draws a token from a
//                         distribution (T > 0), every chunk of the one row
//                         it draws from (§3.1 step 4, §5.2 step (5), §5.3),
//                         handed out from a second counter in the order the
//                         requests' merges publish their rows.
//
// Because row blocks go out request after request, requests complete while
// the stream runs, and the residual work of each request overlaps the rows
// of later ones.  Every byte streams with an evict-first L2 policy, so the
// re-read of a drawn row comes from DRAM (keeping rows, or only every
// request's row 0, resident in L2 measured no faster overall).  No CTA ever
// waits for a specific other CTA: all work is claimed dynamically, so
// progress does not depend on which CTAs are resident.
//
// Roles inside a CTA:
//   claimer lane    claims blocks of work (all the global round trips of
//                   work distribution) and queues them for the producer;
//   producer lane   streams each item of a claimed block into a shared-memory
//                   stage with 1-D TMA bulk copies (logits, plus q for a
//                   residual item) and observes item completions in issue
//                   order through the stage-release barriers;
//   consumer pairs  two warps reduce one item together, each half of it
//                   (chunk statistics or residual sums), and combine;
//   counter warp    adds completed runs of items to the requests' global
//                   arrival counters (a batch of runs at once, one per
//                   lane); a complete count makes a job due;
//   job warp        takes tickets over the jobs (one merge + accept step
//                   per request, one inverse-CDF search per drawn row) and
//                   runs the job it draws once its count is complete.  Jobs
//                   go to whichever CTA asks next, so they run in parallel
//                   across the grid whatever CTA completed the requests.
// Every wait is bounded (about 2 s of %globaltimer); a timeout sets
// SV_FAULT_TIMEOUT and the CTA leaves in order.
#pragma once

#include "sv_device.cuh"
#include "sv_layout.cuh"
#include "sv_resample.cuh"
#include "sv_rowstats.cuh"

namespace sv {

#ifndef SV_PAIRS
#define SV_PAIRS 4
#endif
#ifndef SV_STAGES
#define SV_STAGES 8
#endif
#ifndef SV_ROW_BLOCK
#define SV_ROW_BLOCK 8
#endif
#ifndef SV_RES_BLOCK
#define SV_RES_BLOCK 4
#endif
#ifndef SV_CLAIM_SLOTS
#define SV_CLAIM_SLOTS 1
#endif
#ifndef SV_LOCAL_JOBS_B
#define SV_LOCAL_JOBS_B 1
#endif
#ifndef SV_POLL_NS
#define SV_POLL_NS 0
#endif
#ifndef SV_PREFETCH_NS
#define SV_PREFETCH_NS 3000
#endif
constexpr int kPairs = SV_PAIRS;             // consumer pairs
constexpr int kStages = SV_STAGES;
constexpr int kRowBlock = SV_ROW_BLOCK;      // row-statistics items per claim (base)
// Large batches claim bigger row blocks -- about kRowBlocksPerCta of them per
// CTA, up to kRowBlockMax items -- which halves the row claims of 256 ragged
// requests at V = 151936 (106.2 vs 108.0 us); 128 requests of 6 rows and 64
// of 9 keep the base size (bigger blocks there delay the last merges).
constexpr int kRowBlockMax = 16;
constexpr int kRowBlocksPerCta = 6;
constexpr int kResBlock = SV_RES_BLOCK;      // residual items per claim
// Claimed blocks queued ahead of the producer.  One: a deeper queue holds
// rows (and residual work) claimed early behind a CTA's staged items, so the
// last requests' merges, and the residual work that follows them, start later
// (64 requests of 9 bf16 rows of 128256 logits: 50.2 us with two, 46.3 us
// with one; larger batches unchanged or faster).
constexpr int kClaimSlots = SV_CLAIM_SLOTS;
constexpr unsigned kPollNs = SV_POLL_NS;      // pause between polls of a global flag
// A job warp whose merge is not due this long after it took the ticket
// gathers the merge's draft inputs (ids, uniforms, l(x), q(x)) while it
// waits, so the merge itself needs one wave of loads.  Early merges never
// wait that long; the ones that end the step do.
constexpr uint64_t kPrefetchNs = SV_PREFETCH_NS;
// Batches of up to this many requests run each merge and search in the
// counter warp that completes its input (the kernel's kLocal variant), saving the hand-off to another SM's job
// warp (~1.5 us each) on a step that is one chain of latencies.  With more
// requests one counter warp can complete several and would run their jobs
// in series (measured: B = 1, 25 vs 28 us; B = 8, 40 vs 32 us).
constexpr int kLocalJobsB = SV_LOCAL_JOBS_B;
constexpr int kWarpProducer = 0, kWarpClaimer = 1, kWarpConsumer0 = 2;
constexpr int kWarpCounter = kWarpConsumer0 + 2 * kPairs, kWarpJob = kWarpCounter + 1;
constexpr int kThreads = 32 * (kWarpJob + 1);
#ifndef SV_SMEM_REQ
#define SV_SMEM_REQ 256
#endif
constexpr int kSmemReq = SV_SMEM_REQ;  // requests whose row offsets and scales sit in shared memory
constexpr int kTableWarps = kWarpJob + 1 - kWarpConsumer0;  // warps that build them
constexpr int kTableThreads = 32 * kTableWarps;
constexpr int kScanPer = (kSmemReq + kTableThreads - 1) / kTableThreads;
constexpr uint32_t kRoles = 2 + 2 * kPairs + 2;  // producer, claimer, consumers, counter, job

// Named barrier 1 over the table-building warps.
__device__ __forceinline__ void table_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kTableThreads) : "memory");
}
constexpr int kRunRing = 32;
static_assert(kStages % kPairs == 0, "each consumer pair owns whole stages");
static_assert(kRunRing > kStages + 1, "every open run fits (each holds an unobserved item)");

struct Item {
  int kind;   // 0 row statistics, 1 residual, -1 end of stream
  int c;      // chunk within the row
  int ne;     // elements in the chunk
  int has_q;  // residual item reads a q chunk
  int slot;   // row statistics: padded row index; residual: descriptor slot
  float cs;   // row statistics with tables in global memory: log2(e) / T (0: greedy)
  int b;      // row statistics: request
  int pad;
  Desc d;     // residual item: the row and its statistics
};

// A block of work claimed by the claimer lane.
struct Claim {
  int kind;  // 0 row items [a, a_end), 1 residual chunks [c0, c1) of slot b, -1 end
  uint32_t a, a_end;
  int b, c0, c1;
  int pad[2];
  Desc d;    // residual: the slot's published row
};

// A run of consecutive items of one request (one kind) issued by a CTA.
struct Run {
  int kind;       // 0 row statistics, 1 residual
  int id;         // request (row statistics) or descriptor slot (residual)
  int count;
  int nr;         // rows of the request (row statistics)
  uint32_t last;  // local index of the run's last item
};

// A completed run, handed from the producer lane to the counter warp.
struct Done {
  int kind;  // 0, 1 as in Run; -1 end of stream
  int id;
  int count;
  int nr;
};


constexpr size_t verify_smem_bytes() {
  return static_cast<size_t>(kStages) * kStageBytes + kStages * sizeof(Item) +
         2 * kStages * sizeof(uint64_t);
}

// kLocal: the counter warp runs the jobs it completes (batches of at most
// kLocalJobsB requests); otherwise job warps draw them.
template <typename T, bool kTMA, bool kLocal>
__global__ void __launch_bounds__(kThreads, 1) sv_verify_kernel(Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ SvcQueue<Done> svcq_s;
  __shared__ SvcQueue<Claim, kClaimSlots> clq_s;
  __shared__ float2 xch_s[kStages];     // half 1's partial result of the stage's item
  __shared__ uint64_t xbar_s[kStages];  // ... and the barrier that hands it over
  __shared__ int row_start_s[kSmemReq + 1];
  __shared__ float cs_s[kSmemReq];
  __shared__ int wsum_s[kTableWarps];
  __shared__ Ctl ctl_s;            // the call's counter set, once the header is checked
  __shared__ uint64_t ctl_bar_s;   // completes when ctl_s is written
  __shared__ uint64_t tab_bar_s;   // completes when the shared tables are built
  __shared__ uint32_t err_s;       // this CTA's SV_FAULT_* bits (flushed when it leaves)
  __shared__ uint32_t left_s;      // roles of this CTA that have finished
  auto *svcq = &svcq_s;
  auto *clq = &clq_s;
  Item *info = reinterpret_cast<Item *>(smem + kStages * kStageBytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(info + kStages);
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kStages);
  const uint32_t ctl_bar = smem_addr(&ctl_bar_s), tab_bar = smem_addr(&tab_bar_s);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.gmax + 1;
  constexpr int kRowChunk = Tiling<T>::kRowChunk;
  constexpr int kResChunk = Tiling<T>::kResChunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 2);  // both warps of the owning pair
    }
    for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&xbar_s[s]), 1);
    mbar_init(ctl_bar, 1);
    mbar_init(tab_bar, 1);
    svc_init(svcq);
    svc_init(clq);
    err_s = 0u;
    left_s = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // the inputs, and the workspace as the previous call left it
  // The next call's grid may become resident as CTAs of this one leave; it
  // waits for this grid's completion before it reads anything.
  pdl_launch_dependents();

  uint32_t *err = &err_s;
  const bool uniform = p.lens == nullptr;       // every request has gmax + 1 rows
  const bool smem_req = p.tables_global == 0;  // per-CTA tables in shared memory
  const T *logits = static_cast<const T *>(p.logits);
  auto row_start = [&](int b) {
    return uniform ? b * R : (smem_req ? row_start_s[b] : ld_cg(p.row_start + b));
  };
  auto scale = [&](int b) { return smem_req ? cs_s[b] : ld_cg(p.cs + b); };
  auto wait_ctl = [&]() -> Ctl {  // the call's counter set (ctr null: the wait gave up)
    Ctl c{};
    if (mbar_wait(ctl_bar, 0u, err)) c = ctl_s;
    return c;
  };
  // Each role's lane 0 calls this once when the role is done.  The CTA's
  // last role hands its wait faults to the call's error word and counts the
  // CTA out; the grid's last CTA advances the epoch for the next call.  A
  // fault also withdraws both certificates, so the next call re-clears.
  auto leave = [&]() {
    if (atomicAdd(&left_s, 1u) != kRoles - 1) return;
    const Ctl c = wait_ctl();
    const uint32_t f = atomicOr(&err_s, 0u);
    if (c.ctr && f) atomicOr(c.err, f);
    if (f || !c.ok) {
      st_relaxed64(&p.hdr->ready[0], 0ull);
      st_relaxed64(&p.hdr->ready[1], 0ull);
    }
    if (c.ctr && atomicAdd(&c.ctr->exited, 1u) == gridDim.x - 1)
      st_relaxed(&p.hdr->epoch, c.epoch + 1u);
  };

  if (warp >= kWarpConsumer0) {
    // ----------------------------------------------- per-CTA tables ----
    // Softmax scales (and, for ragged drafts, first rows) of every request,
    // built by the ten warps that do not stream; the producer and claimer
    // start the first block meanwhile.
    const int tt = threadIdx.x - 32 * kWarpConsumer0, tw = warp - kWarpConsumer0;
    uint64_t hdr0 = 0, rdy0 = 0, rdy1 = 0;
    if (warp == kWarpJob && lane == 0)  // the header, in flight during the tables
      read_header(p, hdr0, rdy0, rdy1);
    if (smem_req) {
      for (int b = tt; b < p.B; b += kTableThreads) {
        const float t = __ldg(p.temp + b);
        cs_s[b] = (t > 0.f) ? kLog2e / t : 0.f;
      }
      if (!uniform) {  // exclusive scan of the row counts
        int v[kScanPer], sum = 0;
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) {
          const int b = tt * kScanPer + j;
          v[j] = b < p.B ? request_rows(p, b) : 0;
          sum += v[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += n;
        }
        if (lane == 31) wsum_s[tw] = incl;
        table_sync();
        int run = incl - sum;
        for (int w = 0; w < tw; ++w) run += wsum_s[w];
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) {
          const int b = tt * kScanPer + j;
          if (b < p.B) row_start_s[b] = run;
          run += v[j];
        }
        if (tt == kTableThreads - 1) row_start_s[p.B] = run;
      }
    }
    table_sync();
    if (tt == 0) mbar_arrive(tab_bar);

    if (warp == kWarpJob) {
      // ------------------------------------------ the call's counters ----
      const Ctl c = check_workspace(p, hdr0, rdy0, rdy1, lane, err);
      if (lane == 0) {
        ctl_s = c;
        mbar_arrive(ctl_bar);  // release: ctl_s
      }
      __syncwarp();
    }
  }

  auto search_slot = [&](const Ctl &c, int sl) { search_request<T, kTMA>(p, c, sl, lane); };

  if (warp == kWarpCounter) {
    // --------------------------------------------------- counter warp ----
    // Takes entry k and whatever entries after it are already queued (lane j
    // holds entry k + j), adds all their runs to the global counters at once
    // with one acquire-release add each; the add that completes a count
    // makes that request's merge (or that slot's search) due.
    const Ctl c = wait_ctl();
    for (uint32_t k = 0; c.ok;) {
      if (!mbar_wait_warp(smem_addr(&svcq->full[k % kSvcSlots]), (k / kSvcSlots) & 1u, err))
        break;
      const uint32_t kj = k + lane;
      const bool queued = lane == 0 || mbar_test_wait(smem_addr(&svcq->full[kj % kSvcSlots]),
                                                      (kj / kSvcSlots) & 1u);
      const unsigned qm = __ballot_sync(kFull, queued);
      const int nb = qm == kFull ? 32 : __ffs(~qm) - 1;
      Done e{-2, 0, 0, 0};
      if (lane < nb) e = svcq->slot[kj % kSvcSlots];
      __syncwarp();
      if (lane < nb) mbar_arrive(smem_addr(&svcq->empty[kj % kSvcSlots]));
      k += nb;
      bool last = false;
      if (e.kind >= 0) {
        uint32_t *cnt = e.kind == 0 ? c.k1 + e.id : c.k2 + e.id;
        const uint32_t total = e.kind == 0 ? static_cast<uint32_t>(e.nr * p.C1)
                                           : static_cast<uint32_t>(p.C2);
        // Release: the run's results (observed by the producer); acquire:
        // every earlier run's, when this one completes the count.
        last = atomic_add_acq_rel(cnt, static_cast<uint32_t>(e.count)) + e.count == total;
      }
      // A job warp sees a completed count itself (its acquire load pairs
      // with this add); in the kLocal variant this warp runs the job and
      // flags it taken.  The set's counters are cleared for the call after
      // next by the next call's CTA 0.
      if constexpr (kLocal) {  // run the jobs that complete here, one after another
        if (last) st_relaxed(p.jflag + (e.kind == 0 ? 0 : p.B) + e.id, c.tag | kJobNone);
        for (unsigned lm = __ballot_sync(kFull, last); lm; lm &= lm - 1) {
          const int src = __ffs(lm) - 1;
          const int kind = __shfl_sync(kFull, e.kind, src), id = __shfl_sync(kFull, e.id, src);
          __syncwarp();  // lane src's acquire orders every lane's reads
          if (kind == 0) {
            merge_request<T>(p, c, id, row_start(id + 1) - row_start(id), scale(id), lane, false,
                             DraftIn{});
          } else {
            search_slot(c, id);
          }
        }
      }
      if (__any_sync(kFull, e.kind == -1)) break;
    }
    __syncwarp();
    if (lane == 0) leave();
    return;
  }

  if (warp == kWarpJob) {
    // ------------------------------------------------------- job warp ----
    // Tickets over 2B jobs: job b < B merges request b, job B + s searches
    // slot s.  A ticket waits until its job is due -- its arrival count is
    // complete -- or will never be (a request without rows, a slot left
    // unused, or -- once every request is merged -- a slot never reserved).
    const Ctl c = wait_ctl();
    constexpr bool kCounts = !kLocal;  // poll arrival counters (kLocal: flags)
    const uint32_t njobs = 2u * static_cast<uint32_t>(p.B);
    const uint32_t due = c.tag | kJobDue, none = c.tag | kJobNone;
    for (; c.ok;) {
      // 1 due, 2 none (next ticket), 3 no more jobs or timeout, 4 no rows,
      // 5 gather the draft inputs now
      int state = 0;
      uint32_t h = 0;
      if (lane == 0) {
        h = atomicAdd(&c.ctr->jq_head, 1u);
        if (h >= njobs) state = 3;
        else if (h < static_cast<uint32_t>(p.B) && row_start(h + 1) == row_start(h)) state = 4;
        if (state == 4) fill_bad_request(p, c, static_cast<int>(h));
      }
      h = __shfl_sync(kFull, h, 0);
      state = __shfl_sync(kFull, state, 0);
      const int rows = h < static_cast<uint32_t>(p.B) && state == 0
                           ? row_start(static_cast<int>(h) + 1) - row_start(static_cast<int>(h))
                           : 0;
      bool pre = false, may_pre = rows > 0 && rows <= 32;
      DraftIn pin{};
      const uint64_t t0 = global_timer_ns();
      while (state == 0 || state == 5) {
        if (state == 5) {  // every lane: its draft position's inputs
          pin = load_draft_inputs<T>(p, static_cast<int>(h), rows - 1, scale(static_cast<int>(h)) == 0.f,
                                     lane);
          pre = true;
          may_pre = false;
          state = 0;
        }
        if (lane == 0) {
          // Acquire polls of the flag, or of the arrival counter (no separate
          // fence once the job is seen to be due).
          const bool merge_job = h < static_cast<uint32_t>(p.B);
          const uint32_t *poll = !kCounts ? p.jflag + h
                                 : merge_job ? c.k1 + h
                                             : c.k2 + (h - p.B);
          const uint32_t full = !kCounts ? due
                                : merge_job ? static_cast<uint32_t>(rows * p.C1)
                                            : static_cast<uint32_t>(p.C2);
          const uint32_t skip = kCounts ? kSkipCount : none;
          while (state == 0) {
            // pairs with the counter warp's release (its flag store, or the
            // acquire-release add that completed the count)
            const uint32_t f = ld_acquire(poll);
            const uint64_t dt = global_timer_ns() - t0;
            if (f == full) {
              state = 1;
            } else if (f == skip) {
              state = 2;
            } else if (h >= static_cast<uint32_t>(p.B) && ld_relaxed(&c.ctr->all_merged) != 0u) {
              fence_acq_rel();  // b_reserved is final now
              if (h - p.B >= ld_relaxed(&c.ctr->b_reserved)) state = 3;
            } else if (may_pre && dt > kPrefetchNs) {
              state = 5;
            } else if (dt > kWaitLimitNs) {
              atomicOr(err, SV_FAULT_TIMEOUT);
              state = 3;
            } else if (kPollNs) {
              __nanosleep(kPollNs);
            }
          }
        }
        __syncwarp();  // lane 0's acquire of the flag orders every lane's reads
        state = __shfl_sync(kFull, state, 0);
      }
      if (state == 3) break;
      if (state != 1) continue;
      const int id = static_cast<int>(h);
      if (id < p.B) {
        merge_request<T>(p, c, id, rows, scale(id), lane, pre, pin);
      } else {
        search_slot(c, id - p.B);
      }
    }
    __syncwarp();
    if (lane == 0) leave();
    return;
  }

  if (warp == kWarpClaimer) {
    if (lane != 0) return;
    // -------------------------------------------------- claimer lane ----
    // Residual work is numbered by descriptor slot (merge order): chunk c of
    // slot s is item s * C2 + c.  While this CTA can still claim rows, it
    // takes residual work only from a slot already written, with one
    // compare-and-swap per pass (a lost race falls through to row work, so
    // it never waits).  Once rows are gone it takes tickets from the same
    // counter (atomicAdd: no race to lose), possibly ahead of the slot's
    // reservation, and waits for them; only CTAs without rows wait, so every
    // row is claimed, every request merged and every ticket resolved.  A
    // ticket past the last reserved slot, once every request is merged, ends
    // the stream.  Row blocks are claimed one ahead (the next block's
    // counter add is issued before the current block is queued), so the
    // claim's round trip overlaps the queueing of the block before.  The first block is
    // static (block i of CTA i): it needs no counter, so it goes out before
    // the workspace header is even read.
    bool ok = true;
    if (!uniform && smem_req) ok = mbar_wait(tab_bar, 0u, err);  // ragged: the row table
    const uint32_t n_rows = uniform ? static_cast<uint32_t>(p.B) * R
                                    : static_cast<uint32_t>(row_start(p.B));
    const uint32_t n_row_items = n_rows * static_cast<uint32_t>(p.C1);
    const uint32_t rb_base =
        min(static_cast<uint32_t>(kRowBlock), max(1u, n_row_items / (2u * gridDim.x)));
    const uint32_t rb =
        min(static_cast<uint32_t>(kRowBlockMax),
            max(rb_base, n_row_items / (static_cast<uint32_t>(kRowBlocksPerCta) * gridDim.x)));
    const uint32_t a_dyn = rb * gridDim.x;  // first item handed out by the counter
    const uint32_t C2 = static_cast<uint32_t>(p.C2);
    // Claim sizes: kRowBlock / kResBlock items, fewer when the batch is small
    // (so that its items spread over the grid), and for rows more when it is
    // large.
    const uint32_t spread = 2u * gridDim.x;
    const uint32_t rt =
        min(static_cast<uint32_t>(kResBlock), max(1u, static_cast<uint32_t>(p.B) * C2 / spread));
    uint32_t k = 0;
    auto push = [&](const Claim &cl) { ok = ok && svc_push(clq, k++, cl, err); };
    uint32_t a_cur = rb * blockIdx.x;
    if (ok && a_cur < n_row_items) {
      push(Claim{0, a_cur, min(a_cur + rb, n_row_items), 0, 0, 0, {0, 0}, Desc{}});
      a_cur = n_row_items;  // the next row block comes from the counter
    }
    const Ctl c = wait_ctl();
    ok = ok && c.ok;
    if (ok) a_cur = a_dyn + atomicAdd(&c.ctr->a_next, rb);
    // Slot s: kReadySample (d holds its descriptor) or kReadySkip once
    // written; 0 when it will never be (every request merged, fewer slots
    // reserved) or on a timeout.
    auto await_slot = [&](uint32_t sl, Desc &d) -> uint32_t {
      if (sl >= static_cast<uint32_t>(p.B)) return 0u;  // at most one slot per request
      const uint64_t t0 = global_timer_ns();
      for (;;) {  // relaxed polls of the slot's eight words
        const uint32_t f = desc_poll(p.desc + static_cast<size_t>(sl) * kDescWords, d, c.tag);
        if (f != kPending) return f;
        // All merged: every reservation is visible, b_reserved is final.
        if (ld_relaxed(&c.ctr->all_merged) != 0u) {
          fence_acq_rel();
          if (sl >= ld_relaxed(&c.ctr->b_reserved)) return 0u;
        }
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicOr(err, SV_FAULT_TIMEOUT);
          ok = false;
          return 0u;
        }
        if (kPollNs) __nanosleep(kPollNs);
      }
    };
    bool rows_left = true, more = true;
    while (ok && more) {
      if (rows_left) {
        const uint2 bc = ld_relaxed2(&c.ctr->b_next);  // {b_next, b_reserved}
        const uint32_t sl = bc.x / C2;
        if (sl < bc.y) {
          Desc d;
          const uint32_t f = desc_poll(p.desc + static_cast<size_t>(sl) * kDescWords, d, c.tag);
          const uint32_t s_end = (sl + 1) * C2;
          if (f == kReadySkip) {
            atomicMax(&c.ctr->b_next, s_end);
            continue;
          }
          if (f == kReadySample) {
            const uint32_t want = min(bc.x + rt, s_end);
            if (atomicCAS(&c.ctr->b_next, bc.x, want) == bc.x) {  // d is complete
              const int c0 = static_cast<int>(bc.x - sl * C2);
              push(Claim{1, 0u, 0u, static_cast<int>(sl), c0, c0 + static_cast<int>(want - bc.x),
                         {0, 0}, d});
              continue;
            }
          }
        }
        if (a_cur < n_row_items) {
          const uint32_t a_pre = a_dyn + atomicAdd(&c.ctr->a_next, rb);
          push(Claim{0, a_cur, min(a_cur + rb, n_row_items), 0,
                     0, 0, {0, 0}, Desc{}});
          a_cur = a_pre;
          continue;
        }
        rows_left = false;
      }
      // A ticket: residual items [r, r + rt), slot by slot.
      const uint32_t r = atomicAdd(&c.ctr->b_next, rt);
      for (uint32_t it = r, r_end = r + rt; ok && it < r_end;) {
        const uint32_t sl = it / C2, s_end = (sl + 1) * C2;
        Desc d;
        const uint32_t f = await_slot(sl, d);
        if (f == 0u) {
          more = false;
          break;
        }
        const uint32_t seg_end = min(r_end, s_end);
        if (f == kReadySample) {
          const int c0 = static_cast<int>(it - sl * C2);
          push(Claim{1, 0u, 0u, static_cast<int>(sl), c0, c0 + static_cast<int>(seg_end - it),
                     {0, 0}, d});
        } else {
          atomicMax(&c.ctr->b_next, s_end);  // an unused slot: pass it over
        }
        it = seg_end;
      }
    }
    // The end marker goes out whatever happened: the producer and the
    // consumers stop on it.
    svc_push(clq, k, Claim{-1, 0u, 0u, 0, 0, 0, {0, 0}, Desc{}}, err);
    leave();
    return;
  }

  if (warp == kWarpProducer) {
    if (lane != 0) return;
    // -------------------------------------------------- producer lane ----
// Every logit and q value is streamed with an evict-first L2 policy: the
    // row statistics read each logit once, and keeping rows in L2 for the
    // residual re-read measured slower (65.2 vs 64.1 us for 128 requests of 6
    // bf16 rows of 151936 logits with evict-normal rows, the same with
    // evict-last).
    const uint64_t pol_l = policy_evict_first(), pol_q = pol_l, pol_r = pol_l;
    uint32_t n = 0, m = 0, pushed = 0;  // items issued / observed released; runs handed over
    bool ok = true;
    if (!uniform && smem_req) ok = mbar_wait(tab_bar, 0u, err);  // ragged: the row table

    // Open runs, oldest first (head in registers, the rest in a ring).
    Run head{0, 0, 0, 0, 0u};
    bool has_head = false;
    Run ring[kRunRing];
    int rh = 0, rc = 0;
    auto add_run = [&](const Run &r) {
      if (!has_head) {
        head = r;
        has_head = true;
      } else {
        ring[(rh + rc) % kRunRing] = r;
        ++rc;
      }
    };
    // Item m was released: hand its run over if it was the run's last item.
    auto released = [&]() {
      if (has_head && head.last == m) {
        ok = svc_push(svcq, pushed++, Done{head.kind, head.id, head.count, head.nr}, err);
        if (rc > 0) {
          head = ring[rh];
          rh = (rh + 1) % kRunRing;
          --rc;
        } else {
          has_head = false;
        }
      }
      ++m;
    };
    auto observe_through = [&](uint32_t j) {  // block until items <= j are released
      while (ok && m <= j) {
        ok = mbar_wait(empty0 + 8 * (m % kStages), (m / kStages) & 1u, err);
        if (ok) released();
      }
    };
    auto observe_ready = [&]() {  // take whatever releases have happened
      bool any = false;
      while (ok && m < n && mbar_test_wait(empty0 + 8 * (m % kStages), (m / kStages) & 1u)) {
        released();
        any = true;
      }
      return any;
    };
    auto next_stage = [&]() -> int {  // the stage item n uses, once it is free
      if (n >= kStages) observe_through(n - kStages);
      return static_cast<int>(n % kStages);
    };
    auto request_of_row = [&](int fr) {  // last request whose first row is <= fr
      int lo = 0, hi = p.B;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (row_start(mid) <= fr) lo = mid;
        else hi = mid;
      }
      return lo;
    };

    // Row-statistics items [a, a_end): flat row fr = a / C1, chunk a % C1.
    auto issue_rows = [&](uint32_t a, uint32_t a_end) {
      int fr = static_cast<int>(a / p.C1), c = static_cast<int>(a - fr * p.C1);
      int b = request_of_row(fr), rs = row_start(b), re = row_start(b + 1);
      while (fr >= re) {  // requests without rows share the offset
        rs = re;
        re = row_start(++b + 1);
      }
      // Scales from shared tables are read by the consumers themselves.
      float cs = smem_req ? 0.f : scale(b);
      bool fresh = true;
      for (uint32_t it = a; ok && it < a_end; ++it, ++c) {
        if (c == p.C1) {
          c = 0;
          if (++fr >= re) {
            do {
              rs = re;
              re = row_start(++b + 1);
            } while (fr >= re);
            cs = smem_req ? 0.f : scale(b);
            fresh = true;
          }
        }
        if (fresh) {
          const int run = static_cast<int>(min(a_end, static_cast<uint32_t>(re) * p.C1) - it);
          add_run(Run{0, b, run, re - rs, n + run - 1});
          fresh = false;
        }
        const int s = next_stage();
        if (!ok) return;
        const int slot = b * R + (fr - rs);
        const int e0 = c * kRowChunk, ne = min(kRowChunk, p.V - e0);
        Item &inf = info[s];
        inf.kind = 0;
        inf.c = c;
        inf.ne = ne;
        inf.slot = slot;
        inf.cs = cs;
        inf.b = b;
        if (kTMA) {
          const uint32_t bytes = static_cast<uint32_t>(ne) * sizeof(T);
          mbar_arrive_expect_tx(full0 + 8 * s, bytes);
          tma_load_1d(smem_addr(smem + static_cast<size_t>(s) * kStageBytes),
                      logits + static_cast<size_t>(slot) * p.V + e0, bytes, full0 + 8 * s,
                      pol_l);
        } else {
          mbar_arrive(full0 + 8 * s);
        }
        ++n;
      }
    };

    // Residual chunks [c0, c1) of descriptor slot sl, whose row is d.
    auto issue_residual = [&](int sl, int c0, int c1, const Desc &d) {
      add_run(Run{1, sl, c1 - c0, 0, n + static_cast<uint32_t>(c1 - c0) - 1});
      const bool hq = d.tok >= 0 && p.q != nullptr;
      for (int c = c0; ok && c < c1; ++c) {
        const int s = next_stage();
        if (!ok) return;
        const int e0 = c * kResChunk, ne = min(kResChunk, p.V - e0);
        Item &inf = info[s];
        inf.kind = 1;
        inf.c = c;
        inf.ne = ne;
        inf.has_q = hq ? 1 : 0;
        inf.slot = sl;
        inf.d = d;
        if (kTMA) {
          const uint32_t lb = static_cast<uint32_t>(ne) * sizeof(T);
          const uint32_t qb = hq ? static_cast<uint32_t>(ne) * 4u : 0u;
          uint8_t *st = smem + static_cast<size_t>(s) * kStageBytes;
          mbar_arrive_expect_tx(full0 + 8 * s, lb + qb);
          tma_load_1d(smem_addr(st), logits + static_cast<size_t>(d.slot) * p.V + e0, lb,
                      full0 + 8 * s, pol_r);
          if (hq)
            tma_load_1d(smem_addr(st + kResChunk * sizeof(T)),
                        p.q + (static_cast<size_t>(d.b) * p.gmax + d.k) * p.V + e0, qb,
                        full0 + 8 * s, pol_q);
        } else {
          mbar_arrive(full0 + 8 * s);
        }
        ++n;
      }
    };

    // Stream the claimed blocks; while none is queued, keep handing this
    // CTA's completed runs to the counter warp (other CTAs' tickets may be
    // waiting for the merges they complete).
    for (uint32_t k = 0; ok; ++k) {
      const int i = static_cast<int>(k % kClaimSlots);
      const uint32_t fb = smem_addr(&clq->full[i]), fp = (k / kClaimSlots) & 1u;
      const uint64_t t0 = global_timer_ns();
      while (ok && !mbar_test_wait(fb, fp)) {
        if (!observe_ready()) __nanosleep(64);
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicOr(err, SV_FAULT_TIMEOUT);
          ok = false;
        }
      }
      if (!ok) break;
      const Claim cl = clq->slot[i];
      mbar_arrive(smem_addr(&clq->empty[i]));
      if (cl.kind < 0) break;
      if (cl.kind == 0) issue_rows(cl.a, cl.a_end);
      else issue_residual(cl.b, cl.c0, cl.c1, cl.d);
    }
    // Hand over the last runs, then stop the counter warp and the consumers.
    if (n > 0) observe_through(n - 1);
    svc_push(svcq, pushed, Done{-1, 0, 0, 0}, err);
    for (int w = 0; w < kPairs; ++w, ++n) {
      const int s = static_cast<int>(n % kStages);
      if (!ok && n >= kStages && !mbar_wait(empty0 + 8 * s, ((n / kStages) & 1u) ^ 1u, err))
        break;
      info[s].kind = -1;
      mbar_arrive(full0 + 8 * s);
    }
    leave();
    return;
  }

  // ---------------------------------------------------- consumer pairs ----
  // Pair g takes items g, g + kPairs, ...; warp h of the pair reduces half
  // h of each item and half 1 hands its partial to half 0, which writes the
  // item's result.  Both warps release the stage.  The hand-over slot and
  // its barrier belong to the stage: half 1 writes the slot again only once
  // the stage is refilled, which needs half 0's release (after its read).
  const int cw = warp - kWarpConsumer0, g = cw >> 1, h = cw & 1;
  for (uint32_t n = g;; n += kPairs) {
    const int s = static_cast<int>(n % kStages);
    if (!mbar_wait_warp(full0 + 8 * s, (n / kStages) & 1u, err)) break;
    const Item &inf = info[s];
    const int kind = inf.kind;
    if (kind < 0) break;
    const uint8_t *stage = smem + static_cast<size_t>(s) * kStageBytes;
    const uint32_t xbar = smem_addr(&xbar_s[s]), xpar = (n / kStages) & 1u;
    bool ok = true;
    if (kind == 0) {
      const int c = inf.c, ne = inf.ne, slot = inf.slot;
      const float cs = smem_req ? cs_s[inf.b] : inf.cs;
      const int ne0 = half0_len(ne);
      const int off = h ? ne0 : 0, len = h ? ne - ne0 : ne0;
      ChunkStat st;
      if (kTMA) {
        st = chunk_stats_smem(reinterpret_cast<const T *>(stage) + off, len, cs, lane);
      } else {
        st = chunk_stats_global<T>(logits + static_cast<size_t>(slot) * p.V, c * kRowChunk + off,
                                   len, cs, lane);
      }
      if (cs == 0.f && __float_as_int(st.v) != 0x7fffffff)
        st.v = __int_as_float(__float_as_int(st.v) + off);
      if (h == 1) {
        __syncwarp();
        if (lane == 0) {
          xch_s[s] = make_float2(st.m, st.v);
          mbar_arrive(xbar);  // release: the partial
        }
      } else {
        ok = mbar_wait_warp(xbar, xpar, err);
        if (ok) {
          const float2 o = xch_s[s];
          st = combine_halves(st, ChunkStat{o.x, o.y}, cs);
          if (cs == 0.f && __float_as_int(st.v) != 0x7fffffff)
            st.v = __int_as_float(__float_as_int(st.v) + c * kRowChunk);
          if (lane == 0) p.part1[static_cast<size_t>(slot) * p.C1 + c] = Part{st.m, st.v};
        }
      }
    } else {
      const Desc d = inf.d;
      const int c = inf.c;
      const int sl = inf.slot;
      const float2 part =
          chunk_resid<T, kTMA>(p, d, sl, c, inf.ne, inf.has_q != 0, stage, h, lane);
      if (h == 1) {
        __syncwarp();
        if (lane == 0) {
          xch_s[s] = part;
          mbar_arrive(xbar);
        }
      } else {
        ok = mbar_wait_warp(xbar, xpar, err);
        if (ok && lane == 0) {
          const float2 o = xch_s[s];
          p.csum[static_cast<size_t>(sl) * p.C2 + c] =
              make_float2(__fadd_rn(part.x, o.x), __fadd_rn(part.y, o.y));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);  // release: publishes the item's results
    if (!ok) break;
  }
  __syncwarp();
  if (lane == 0) leave();
}

}  // namespace sv
