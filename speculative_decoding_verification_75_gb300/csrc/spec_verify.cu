// spec_verify.cu -- C ABI of the GB300 speculative-decoding verification
// library: argument checks, workspace carving and the launches.
//
//   kernel 0  sv_prepare_kernel  only for batches of more than kSmemReq
//                                requests (row offsets and softmax scales in
//                                global memory) or when the caller asks for
//                                the acceptance histogram (its reset)
//   kernel 1  sv_verify_kernel   persistent: softmax statistics of every row,
//                                accept test and first rejection per request,
//                                residual / bonus draw for sampled requests
//
// Both are launched with programmatic stream serialisation, so that a
// launch and its prologue overlap the end of the grid before it.  Kernel 1
// comes in a TMA variant (rows start on 16-byte boundaries) and a plain-load
// variant for any other alignment.  It keeps the workspace ready for the
// next call itself (counter sets alternate by call, see sv_layout.cuh), so
// a call is one launch.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>

#include "spec_verify.h"
#include "sv_device.cuh"
#include "sv_layout.cuh"
#include "sv_kv.cuh"
#include "sv_cluster.cuh"
#include "sv_prepare.cuh"
#include "sv_verify.cuh"

namespace sv {

// Self-test of the bounded waits: an mbarrier phase that nobody completes
// and a device flag that nobody sets, each waited for with a short limit.
// Both must give up, set SV_FAULT_TIMEOUT and let the kernel end.
__global__ void sv_selftest_wait_kernel(uint32_t *word, const uint32_t *never,
                                        uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  if (!mbar_wait_slow(smem_addr(&bar), 0u, word, limit_ns)) atomicOr(word, 0x1u);
  const uint64_t t0 = global_timer_ns();
  while (ld_relaxed(never) == 0u) {
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(word, SV_FAULT_TIMEOUT | 0x2u);
      break;
    }
    __nanosleep(256);
  }
}

namespace {

constexpr int kMaxDevices = 64;
constexpr int kClusterMaxB = 32;  // batches up to this size may take the cluster path
std::atomic<int> g_small_batch_path{1};  // sv_set_small_batch_path

bool sizes_ok(int B, int gmax, int V) {
  if (B < 0 || gmax < 0 || V < 1) return false;
  const long long rows = static_cast<long long>(B) * (gmax + 1);
  return rows < INT_MAX && static_cast<long long>(gmax) * V < (1ll << 62);
}

bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Raise the dynamic shared-memory limit of a kernel once per device.
template <typename K>
cudaError_t ensure_smem(K kernel, size_t bytes, std::atomic<uint64_t> &done, int dev) {
  const uint64_t bit = 1ull << (dev % kMaxDevices);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const Params &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// ------------------------------------------------ small-batch path ----
// One cluster of CS CTAs per request (sv_cluster.cuh), when the whole batch
// fits on the GPU at once: B clusters co-resident, every row slice of a
// request (plus its q slice) in one CTA's shared memory, gamma_max < 16,
// rows aligned for TMA.
constexpr size_t kClusterSmemMax = 220 * 1024;
constexpr size_t kClusterSmemStep = 8 * 1024;
constexpr int kClusterSizes[3] = {16, 12, 8};

// Clusters of cs CTAs with smem bytes of dynamic shared memory each that can
// be resident together, queried once per device, element type, cluster size
// and 8 KiB class of the footprint (the class's upper end: conservative).
template <typename T>
int cluster_capacity(int dev, int cs_index, size_t smem) {
  constexpr int kClasses = static_cast<int>(kClusterSmemMax / kClusterSmemStep);
  static std::atomic<int> cache[kMaxDevices][3][kClasses];  // value + 1
  const int cls = static_cast<int>((smem + kClusterSmemStep - 1) / kClusterSmemStep) - 1;
  if (cls < 0 || cls >= kClasses) return 0;
  std::atomic<int> &slot = cache[dev % kMaxDevices][cs_index][cls];
  int v = slot.load(std::memory_order_acquire);
  if (v > 0) return v - 1;
  const int cs = kClusterSizes[cs_index];
  int n = 0;
  auto *k = sv_cluster_kernel<T>;
  bool ok = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kClusterSmemMax)) == cudaSuccess;
  if (ok && cs > 8)
    ok = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(cls + 1) * kClusterSmemStep;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a refused size only means: not this path
  slot.store(n + 1, std::memory_order_release);
  return n;
}

// Launches the cluster kernel if the batch qualifies (the largest cluster
// size whose footprint fits and whose clusters can all be resident); false
// otherwise.
template <typename T>
bool try_cluster(const Params &p, cudaStream_t st, int dev, sv_status *status) {
  if (p.gmax + 1 > kCMaxRows) return false;
  for (int ci = 0; ci < 3; ++ci) {
    const int cs = kClusterSizes[ci];
    const int W = (p.V + cs - 1) / cs;
    const int Wr = (W + 7) / 8 * 8;  // 16-byte aligned slices (bf16 and fp32)
    const size_t smem = cluster_smem_bytes(p.gmax + 1, Wr, sizeof(T));
    if (smem > kClusterSmemMax || cluster_capacity<T>(dev, ci, smem) < p.B) continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.B * cs));
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    *status = cudaLaunchKernelEx(&cfg, sv_cluster_kernel<T>, p, Wr) == cudaSuccess ? SV_OK
                                                                                   : SV_ERR_CUDA;
    return true;
  }
  return false;
}

template <typename T, bool kTMA>
sv_status launch_all(Params &p, cudaStream_t st, int dev, int nsm) {
  static std::atomic<uint64_t> smem_done{0}, smem_done_local{0};
  p.C1 = div_up(p.V, Tiling<T>::kRowChunk);
  p.C2 = div_up(p.V, Tiling<T>::kResChunk);
  p.nseg = p.C2 * Tiling<T>::kSegPerChunk;

  const bool local = p.B <= kLocalJobsB;
  auto *kv = local ? sv_verify_kernel<T, kTMA, true> : sv_verify_kernel<T, kTMA, false>;
  const size_t smem = verify_smem_bytes();
  if (ensure_smem(kv, smem, local ? smem_done_local : smem_done, dev) != cudaSuccess)
    return SV_ERR_CUDA;

  p.tables_global = p.B > kSmemReq ? 1 : 0;
  const bool small = kTMA && p.B <= kClusterMaxB &&
                     g_small_batch_path.load(std::memory_order_relaxed) != 0;
  if ((p.tables_global || p.diag.accept_hist) && !small) {
    if (launch_pdl(sv_prepare_kernel, dim3(1), dim3(kPrepThreads), 0, st, p) != cudaSuccess)
      return SV_ERR_CUDA;
  }
  if (small) {
    Params pc = p;
    pc.tables_global = 0;  // the cluster kernel needs no tables
    if (pc.diag.accept_hist &&
        launch_pdl(sv_prepare_kernel, dim3(1), dim3(kPrepThreads), 0, st, pc) != cudaSuccess)
      return SV_ERR_CUDA;
    sv_status s = SV_OK;
    if (try_cluster<T>(pc, st, dev, &s)) return s;
    if (p.tables_global &&
        launch_pdl(sv_prepare_kernel, dim3(1), dim3(kPrepThreads), 0, st, p) != cudaSuccess)
      return SV_ERR_CUDA;
  }

  const long long max_items = static_cast<long long>(p.B) * (p.gmax + 1) * p.C1;
  const int grid = static_cast<int>(max_items < nsm ? max_items : nsm);
  if (launch_pdl(kv, dim3(grid), dim3(kThreads), smem, st, p) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

sv_status run(const void *logits, sv_dtype dtype, const int32_t *ids, const float *q,
              const float *u_acc, const float *u_smp, const float *temp,
              const int32_t *lens, int B, int gmax, int V, int32_t *out_tokens,
              int32_t *out_nacc, void *ws, size_t ws_bytes, sv_stream_t stream,
              const sv_diag *diag) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_UNSUPPORTED_DTYPE;
  if (!sizes_ok(B, gmax, V)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !u_smp || !temp || !out_tokens || !out_nacc || !ws)
    return SV_ERR_INVALID_ARG;
  if (gmax > 0 && (!ids || !u_acc)) return SV_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return SV_ERR_INVALID_ARG;
  const size_t esz = dtype == SV_BF16 ? 2 : 4;
  if (!aligned(logits, esz) || (q && !aligned(q, 4))) return SV_ERR_INVALID_ARG;
  const Layout L = make_layout(B, gmax, V);
  if (ws_bytes < L.total) return SV_ERR_WORKSPACE_TOO_SMALL;

  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SV_ERR_CUDA;

  uint8_t *w = static_cast<uint8_t *>(ws);
  Params p{};
  p.logits = logits;
  p.ids = ids;
  p.q = q;
  p.u_acc = u_acc;
  p.u_smp = u_smp;
  p.temp = temp;
  p.lens = lens;
  p.B = B;
  p.gmax = gmax;
  p.V = V;
  p.out_tokens = out_tokens;
  p.out_nacc = out_nacc;
  if (diag) p.diag = *diag;
  p.hdr = reinterpret_cast<Header *>(w + L.hdr);
  p.row_start = reinterpret_cast<int *>(w + L.row_start);
  p.cs = reinterpret_cast<float *>(w + L.cs);
  p.k1_cnt = reinterpret_cast<uint32_t *>(w + L.k1_cnt);
  p.k2_cnt = reinterpret_cast<uint32_t *>(w + L.k2_cnt);
  p.desc = reinterpret_cast<uint64_t *>(w + L.desc);
  p.jflag = reinterpret_cast<uint32_t *>(w + L.jflag);
  p.part1 = reinterpret_cast<Part *>(w + L.part1);
  p.csum = reinterpret_cast<float2 *>(w + L.csum);
  p.ssum = reinterpret_cast<float2 *>(w + L.ssum);

  // TMA bulk copies need 16-byte aligned rows: the base pointers and the
  // row pitch of the logits (and of q, when present).
  const bool tma = aligned(logits, 16) && (static_cast<size_t>(V) * esz) % 16 == 0 &&
                   (!q || (aligned(q, 16) && (static_cast<size_t>(V) * 4) % 16 == 0));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    return tma ? launch_all<__nv_bfloat16, true>(p, st, dev, nsm)
               : launch_all<__nv_bfloat16, false>(p, st, dev, nsm);
  return tma ? launch_all<float, true>(p, st, dev, nsm)
             : launch_all<float, false>(p, st, dev, nsm);
}

}  // namespace
}  // namespace sv

extern "C" {

size_t sv_workspace_bytes(int B, int gamma_max, int V) {
  if (!sv::sizes_ok(B, gamma_max, V)) return 0;
  return sv::make_layout(B, gamma_max, V).total;
}

sv_status spec_verify(const void *target_logits, sv_dtype logits_dtype,
                      const int32_t *draft_token_ids, const float *draft_probs,
                      const float *uniforms_accept, const float *uniforms_sample,
                      const float *temperature, const int32_t *draft_lens, int B,
                      int gamma_max, int V, int32_t *out_tokens, int32_t *out_num_accepted,
                      void *workspace, size_t workspace_bytes, sv_stream_t stream) {
  return sv::run(target_logits, logits_dtype, draft_token_ids, draft_probs, uniforms_accept,
                 uniforms_sample, temperature, draft_lens, B, gamma_max, V, out_tokens,
                 out_num_accepted, workspace, workspace_bytes, stream, nullptr);
}

sv_status spec_verify_diag(const void *target_logits, sv_dtype logits_dtype,
                           const int32_t *draft_token_ids, const float *draft_probs,
                           const float *uniforms_accept, const float *uniforms_sample,
                           const float *temperature, const int32_t *draft_lens, int B,
                           int gamma_max, int V, int32_t *out_tokens,
                           int32_t *out_num_accepted, void *workspace,
                           size_t workspace_bytes, sv_stream_t stream, const sv_diag *diag) {
  return sv::run(target_logits, logits_dtype, draft_token_ids, draft_probs, uniforms_accept,
                 uniforms_sample, temperature, draft_lens, B, gamma_max, V, out_tokens,
                 out_num_accepted, workspace, workspace_bytes, stream, diag);
}

sv_status sv_last_error(const void *workspace, sv_stream_t stream, uint32_t *out_word) {
  if (!workspace) return SV_ERR_INVALID_ARG;
  // The header's first words: the epoch (calls completed) and the error
  // words of the two call parities; the last call ran with epoch - 1.
  uint32_t head[3] = {0, 0, 0};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(head, workspace, sizeof head, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SV_ERR_CUDA;
  const uint32_t word = head[1 + ((head[0] - 1u) & 1u)];
  if (out_word) *out_word = word;
  if (word & SV_FAULT_TIMEOUT) return SV_ERR_TIMEOUT;
  if (word) return SV_ERR_BAD_INPUT_DATA;
  return SV_OK;
}

sv_status sv_kv_rollback(const int32_t *num_accepted, const int32_t *draft_lens,
                         int32_t *seq_lens, int32_t *block_tables, int B, int gamma_max,
                         int max_blocks, int block_size, int32_t *free_list,
                         int32_t *free_count, int free_capacity, uint32_t *status,
                         sv_stream_t stream) {
  if (B < 0 || gamma_max < 0 || max_blocks < 0 || block_size < 1 || free_capacity < 0)
    return SV_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * max_blocks >= INT_MAX ||
      static_cast<long long>(max_blocks) * block_size >= INT_MAX)
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!num_accepted || !seq_lens || !block_tables || !free_count ||
      (free_capacity > 0 && !free_list))
    return SV_ERR_INVALID_ARG;
  sv::KvParams kp{num_accepted, draft_lens, seq_lens, block_tables, B, gamma_max, max_blocks,
                  block_size, free_list, free_count, free_capacity, status};
  const int grid = (B + sv::kKvThreads - 1) / sv::kKvThreads;
  sv::sv_kv_rollback_kernel<<<grid, sv::kKvThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(kp);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_selftest_wait_timeout(uint32_t *word, const uint32_t *never_set,
                                    unsigned limit_us, sv_stream_t stream) {
  if (!word || !never_set || limit_us == 0 || limit_us > 1000000u) return SV_ERR_INVALID_ARG;
  sv::sv_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      word, never_set, static_cast<uint64_t>(limit_us) * 1000u);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int sv_set_small_batch_path(int enabled) {
  return sv::g_small_batch_path.exchange(enabled ? 1 : 0);
}

const char *sv_status_string(sv_status status) {
  switch (status) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: invalid argument";
    case SV_ERR_UNSUPPORTED_DTYPE: return "SV_ERR_UNSUPPORTED_DTYPE: logits dtype not fp32/bf16";
    case SV_ERR_WORKSPACE_TOO_SMALL: return "SV_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: CUDA runtime call or launch failed";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded device wait gave up";
    case SV_ERR_BAD_INPUT_DATA: return "SV_ERR_BAD_INPUT_DATA: a request had invalid data";
  }
  return "unknown sv_status";
}

// ------------------------------------------------ allocation-free variant ----
// For callers that cannot allocate device memory: the workspace lives in one
// file-scope device array instead of caller memory.  Host code never uses the
// array's name as an address (on the host it is only a stand-in symbol); its
// device address is looked up once per device with cudaGetSymbolAddress.

namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];
std::atomic<void *> g_noalloc_addr[sv::kMaxDevices];

// Device address of the scratch array on the current device (looked up on
// the first call per device, that device being current).
sv_status noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= sv::kMaxDevices) return SV_ERR_CUDA;
  void *ptr = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SV_ERR_CUDA;
    g_noalloc_addr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return SV_OK;
}
}  // namespace

sv_status spec_verify_noalloc(const void *target_logits, sv_dtype logits_dtype,
                              const int32_t *draft_token_ids, const float *draft_probs,
                              const float *uniforms_accept, const float *uniforms_sample,
                              const float *temperature, const int32_t *draft_lens, int B,
                              int gamma_max, int V, int32_t *out_tokens,
                              int32_t *out_num_accepted, sv_stream_t stream) {
  if (logits_dtype != SV_F32 && logits_dtype != SV_BF16) return SV_ERR_UNSUPPORTED_DTYPE;
  if (!sv::sizes_ok(B, gamma_max, V)) return SV_ERR_INVALID_ARG;
  if (sv::make_layout(B, gamma_max, V).total > SV_NOALLOC_SCRATCH_BYTES)
    return SV_ERR_WORKSPACE_TOO_SMALL;
  if (B == 0) return SV_OK;
  void *scratch = nullptr;
  const sv_status st = noalloc_scratch(&scratch);
  if (st != SV_OK) return st;
  return sv::run(target_logits, logits_dtype, draft_token_ids, draft_probs, uniforms_accept,
                 uniforms_sample, temperature, draft_lens, B, gamma_max, V, out_tokens,
                 out_num_accepted, scratch, SV_NOALLOC_SCRATCH_BYTES, stream, nullptr);
}

}  // extern "C"
