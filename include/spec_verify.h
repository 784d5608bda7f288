/*
 * spec_verify.h -- C ABI of the GB300 speculative-decoding verification
 * library (libspecverify.so).
 *
 * The operation is the verification step of speculative decoding as the
 * tutorial page at http://www.dpshk.com/news/5598276/ ("P3"; its HTML title,
 * 企业官网建设流程全解析, is unrelated to its content) defines it:
 *   P3 §3.1 steps 2-4 and §5.2 steps (1)-(5):
 *     p_i   = softmax(target_logits[b, i, :] / T_b)              (i <= g_b)
 *     a_i   = min(1, p_i(x_i) / max(q_i(x_i), 1e-10))            (i <  g_b)
 *     keep  x_i while u_i < a_i; k_b = first i with u_i >= a_i (else g_b)
 *     token at k_b: drawn from (p_k - q_k)_+ / sum (p_k - q_k)_+ on a
 *     rejection, from p_{g_b} (the bonus row, §5.3) when all are kept.
 *   Draws are inverse-CDF draws on the caller's uniform u_s[b]: the token is
 *   the smallest j whose inclusive prefix sum of the (unnormalised) weights
 *   exceeds u_s[b] times their total, so a token without weight is never
 *   drawn; where binary32 rounding leaves u_s[b] times the total at or past
 *   the summed weights, the last token with positive weight.  An empty
 *   residual (every (p - q)_+ zero) draws from p_k instead.  T_b = 0 is
 *   greedy decoding (P3 §8,
 *   pitfall 2): p is one-hot at the lowest-index maximum logit.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers to dense row-major arrays,
 *     owned by the caller; the library allocates nothing and keeps no state
 *     between calls.  The caller also owns the workspace and the stream.
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream).  Host-side argument checks return an error before anything is
 *     enqueued; a failed launch returns SV_ERR_CUDA.
 *   - spec_verify and its variants launch their kernels as programmatic
 *     dependent launches: their first kernel waits for the completion of
 *     whatever precedes it on the stream before it touches memory, and the
 *     last one allows the next kernel on the stream to be scheduled early.
 *     A kernel launched after it WITH programmatic stream serialization must
 *     wait for its prerequisites (griddepcontrol.wait /
 *     cudaGridDependencySynchronize) before reading the outputs; ordinary
 *     launches, copies and events are unaffected.
 *   - Invalid per-request DATA (a draft length outside [0, gamma_max], a
 *     temperature that is negative, NaN, inf or subnormal, a draft token id
 *     outside [0, V), a uniform outside [0, 1), a non-finite softmax
 *     normaliser) never traps: that request gets out_num_accepted = -1 and an
 *     all -1 token row, other requests are unaffected, and the matching
 *     SV_BAD_* bit is set in the workspace's error word (sv_last_error).
 *   - Outputs must not alias inputs or the workspace.  Calls that share one
 *     workspace must be ordered on one stream.
 *   - Logits must be finite for greedy rows (T = 0); for T > 0 a NaN or +inf
 *     logit marks the request bad, and -inf logits are allowed (masked
 *     tokens) as long as each row has a finite maximum.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SV_API __attribute__((visibility("default")))
#else
#define SV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (a CUstream handle); NULL = default stream. */
typedef struct CUstream_st *sv_stream_t;

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,        /* NULL pointer, negative size, misaligned
                                      workspace, sizes beyond int32 indexing */
    SV_ERR_UNSUPPORTED_DTYPE = 2,  /* logits_dtype is not SV_F32 / SV_BF16 */
    SV_ERR_WORKSPACE_TOO_SMALL = 3,/* workspace_bytes < sv_workspace_bytes() */
    SV_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed */
    SV_ERR_TIMEOUT = 5,            /* a bounded device-side wait ran out */
    SV_ERR_BAD_INPUT_DATA = 6      /* some request had invalid data */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Bits of the device error word read back by sv_last_error(). */
#define SV_BAD_DRAFT_LEN 0x1u    /* draft_lens[b] outside [0, gamma_max]     */
#define SV_BAD_TEMPERATURE 0x2u  /* T negative, NaN, inf or subnormal       */
#define SV_BAD_TOKEN 0x4u        /* a draft token id outside [0, V)         */
#define SV_BAD_U_ACCEPT 0x8u     /* an acceptance uniform outside [0, 1)    */
#define SV_BAD_U_SAMPLE 0x10u    /* the sampling uniform outside [0, 1)     */
#define SV_BAD_NORMALISER 0x20u  /* non-finite softmax normaliser (T > 0),
                                    or a row maximum m with
                                    |m * log2(e) / T| >= 2^24 in binary32
                                    (T too small to form p's exponents)    */
#define SV_FAULT_TIMEOUT 0x10000u/* a bounded wait inside a kernel gave up  */

/*
 * Workspace size in bytes for a batch of B requests with up to gamma_max
 * drafts each over a V-token vocabulary (any logits dtype).  The workspace
 * must be device memory aligned to 256 bytes.  It needs no initialisation:
 * each call leaves it ready for the next (its work counters alternate
 * between two sets by call), and a call that finds it not ready -- fresh or
 * foreign bytes, another (B, gamma_max, V), a call that gave up -- clears it
 * first.  Returns 0 for invalid sizes.
 */
SV_API size_t sv_workspace_bytes(int B, int gamma_max, int V);

/*
 * One verification step for a batch (P3 §3.1, §5.2, §5.3).
 *
 *   target_logits    [B, gamma_max+1, V]  logits_dtype (fp32 or bf16).  Row
 *                    i of request b is the target model's output after the
 *                    prefix and drafts x_0..x_{i-1}; row g_b is the bonus row.
 *                    Rows past g_b are never read.
 *   draft_token_ids  [B, gamma_max] int32: x_i, the drafted tokens.
 *   draft_probs      [B, gamma_max, V] fp32: q_i, the draft model's
 *                    distribution at each drafted position, already at the
 *                    draft's own temperature.  NULL means deterministic
 *                    drafts (prompt lookup, P3 §7): q_i is one-hot at x_i.
 *   uniforms_accept  [B, gamma_max] fp32 in [0, 1): the accept test's dice.
 *   uniforms_sample  [B] fp32 in [0, 1): the resample or bonus draw.
 *   temperature      [B] fp32: T_b >= 0, divides the target logits; 0 is
 *                    greedy.
 *   draft_lens       [B] int32 g_b in [0, gamma_max], or NULL: every request
 *                    drafts gamma_max tokens.  g_b = 0 is plain sampling from
 *                    row 0.
 *   B, gamma_max, V  B >= 0 (0 is a no-op), gamma_max >= 0, V >= 1, with
 *                    B*(gamma_max+1) and V below 2^31.
 *   out_tokens       [B, gamma_max+1] int32: x_0..x_{k-1}, then the
 *                    resampled, bonus or argmax token at position k, then -1.
 *   out_num_accepted [B] int32: k_b, or -1 for a request with invalid data.
 *   workspace        device scratch of at least sv_workspace_bytes(B,
 *                    gamma_max, V) bytes, 256-byte aligned.
 *
 * Arithmetic is fp32 (bf16 logits widen exactly); accept decisions and drawn
 * tokens equal an exact-arithmetic evaluation except where the decision
 * margin (|u - a|, or the distance of u*S to a CDF edge) is of the order of
 * fp32 rounding.  Results are deterministic for identical inputs.
 */
SV_API sv_status spec_verify(const void *target_logits, sv_dtype logits_dtype,
                      const int32_t *draft_token_ids, const float *draft_probs,
                      const float *uniforms_accept,
                      const float *uniforms_sample, const float *temperature,
                      const int32_t *draft_lens, int B, int gamma_max, int V,
                      int32_t *out_tokens, int32_t *out_num_accepted,
                      void *workspace, size_t workspace_bytes,
                      sv_stream_t stream);

/*
 * Optional diagnostic outputs (device pointers; any may be NULL).  Slots a
 * request does not use hold NaN (floats), 2 (flags) or -1 (indices).
 */
typedef struct {
    float *p_tok;        /* [B, gamma_max]   p_i(x_i)                        */
    float *q_tok;        /* [B, gamma_max]   q_i(x_i) before the 1e-10 clamp */
    float *accept_prob;  /* [B, gamma_max]   a_i                             */
    uint8_t *flags;      /* [B, gamma_max]   1 accepted, 0 rejected (every
                                             position < g_b is evaluated)    */
    float *row_max;      /* [B, gamma_max+1] max_j logit                     */
    float *row_sum;      /* [B, gamma_max+1] sum_j exp((l_j - max) / T); 1
                                             for greedy rows                 */
    int32_t *row_argmax; /* [B, gamma_max+1] lowest argmax (greedy rows
                                             only; -1 for T > 0 rows)        */
    float *resid_mass;   /* [B] S = sum_j (p_k - q_k)_+ of the draw (NaN for
                                greedy requests)                             */
    int32_t *accept_hist;/* [gamma_max + 2] acceptance statistics of the
                            batch in the same pass (P3 §6.2 logs the
                            acceptance rate; §3.3 gives its expectation):
                            accept_hist[j] = requests with num_accepted == j
                            (j <= gamma_max), accept_hist[gamma_max + 1] =
                            requests with invalid data.  Position i was
                            accepted by sum_{j > i} accept_hist[j] requests.
                            Zeroed by the call; no extra pass over the
                            logits.                                          */
} sv_diag;

/* spec_verify plus the diagnostic outputs in `diag` (may be NULL). */
SV_API sv_status spec_verify_diag(const void *target_logits, sv_dtype logits_dtype,
                           const int32_t *draft_token_ids,
                           const float *draft_probs,
                           const float *uniforms_accept,
                           const float *uniforms_sample,
                           const float *temperature, const int32_t *draft_lens,
                           int B, int gamma_max, int V, int32_t *out_tokens,
                           int32_t *out_num_accepted, void *workspace,
                           size_t workspace_bytes, sv_stream_t stream,
                           const sv_diag *diag);

/*
 * Self-test of failure detection without a GPU fault: launches one small
 * kernel that waits, with a limit of `limit_us` microseconds (1 .. 10^6),
 * for an mbarrier phase that nobody completes and for the device word
 * `never_set` (the caller keeps it 0).  Both waits must give up: the kernel
 * ORs SV_FAULT_TIMEOUT | 0x1 (the mbarrier wait) and 0x2 (the flag wait)
 * into the device word `word` (the caller zeroes it) and ends; the context
 * stays usable.  The verification kernels use the same waits with a ~2 s
 * limit.  Asynchronous on `stream`.
 */
SV_API sv_status sv_selftest_wait_timeout(uint32_t *word, const uint32_t *never_set,
                                          unsigned limit_us, sv_stream_t stream);

/*
 * KV rollback hand-off after verification (P3 §5.4: the KV of the drafted
 * tokens is written first and marked tentative; after verification the cache
 * is cut at num_accepted and the blocks past the cut go back to the block
 * pool; the corrected token's KV is computed by the next step).
 *
 * For a paged KV cache, per request b with L = seq_lens[b] committed tokens
 * before the drafts, g = draft_lens[b] (NULL: gamma_max) drafts at positions
 * L .. L+g-1, and k = num_accepted[b] kept (as returned by spec_verify;
 * k < 0, an invalid request, keeps none):
 *   the entries j in [ceil((L+k)/block_size), ceil((L+g)/block_size)) of
 *   block_tables[b] that hold a block id (>= 0) are appended to free_list at
 *   free_list[*free_count ...] (in no particular order) and set to -1, and
 *   seq_lens[b] becomes L + k.
 * Device pointers: num_accepted, draft_lens [B]; seq_lens [B] (in/out);
 * block_tables [B, max_blocks] (in/out); free_list [free_capacity];
 * free_count a device int32 (in/out); status an optional device uint32 that
 * receives SV_KV_* bits (OR-ed; the caller zeroes it).  Asynchronous on
 * `stream`; allocates nothing.
 * Problems in the data never fault: a request with an invalid draft length
 * or a negative length is left unchanged (SV_KV_BAD_LENGTH); entries past
 * max_blocks are not touched (SV_KV_TABLE_SHORT); an entry that should hold
 * a block but is -1 is skipped (SV_KV_MISSING_BLOCK); a block that does not
 * fit in the free list stays in the table, *free_count stops at
 * free_capacity (SV_KV_FREE_LIST_FULL) and seq_lens is still updated.
 * Returns SV_ERR_INVALID_ARG for negative sizes, block_size < 1, NULL
 * required pointers or B * max_blocks beyond int32 indexing; SV_OK for
 * B == 0 (nothing launched).
 */
#define SV_KV_FREE_LIST_FULL 0x1u
#define SV_KV_MISSING_BLOCK 0x2u
#define SV_KV_BAD_LENGTH 0x4u
#define SV_KV_TABLE_SHORT 0x8u
SV_API sv_status sv_kv_rollback(const int32_t *num_accepted, const int32_t *draft_lens,
                                int32_t *seq_lens, int32_t *block_tables, int B,
                                int gamma_max, int max_blocks, int block_size,
                                int32_t *free_list, int32_t *free_count,
                                int free_capacity, uint32_t *status, sv_stream_t stream);

/*
 * Reads the error word of the last call that used `workspace` (synchronises
 * `stream`).  *out_word (may be NULL) receives the SV_BAD_* / SV_FAULT_*
 * bits.  Returns SV_ERR_TIMEOUT if a bounded wait gave up, else
 * SV_ERR_BAD_INPUT_DATA if any request had invalid data, else SV_OK
 * (SV_ERR_CUDA if the copy fails, SV_ERR_INVALID_ARG for a NULL workspace).
 */
SV_API sv_status sv_last_error(const void *workspace, sv_stream_t stream,
                        uint32_t *out_word);

/*
 * Small batches (B <= 32, gamma_max < 16, rows on 16-byte boundaries, a
 * request's row slices fitting one CTA's shared memory, and every cluster
 * resident at once) run on the cluster path: one thread-block cluster per
 * request whose CTAs split the vocabulary and exchange their statistics
 * through distributed shared memory.  Larger batches run the persistent
 * kernel.  Both compute the same step; sv_set_small_batch_path(0) sends
 * every batch to the persistent kernel (process-wide, e.g. to compare the
 * two), 1 restores the default.  Returns the previous setting.
 */
SV_API int sv_set_small_batch_path(int enabled);

/* Static, human-readable name of a status code. */
SV_API const char *sv_status_string(sv_status status);

/*
 * Allocation-free variant of spec_verify.  The tutorial page has no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- code running inside a CUDA-graph-driven or real-time
 * serving loop that forbids allocation on its hot path, plugins handed a
 * device context but no allocator, or C callers without a CUDA memory
 * manager -- and so cannot provide the workspace spec_verify needs.
 *
 * Instead of a caller-provided workspace it uses one scratch array of
 * SV_NOALLOC_SCRATCH_BYTES bytes that the library defines in device memory
 * (a file-scope __device__ array: every GPU that loads the library keeps it
 * until the process exits).  Everything else -- inputs, outputs, stream,
 * results -- is as for spec_verify.
 *
 *   - Sizes whose workspace, sv_workspace_bytes(B, gamma_max, V), exceeds
 *     SV_NOALLOC_SCRATCH_BYTES are rejected with SV_ERR_WORKSPACE_TOO_SMALL
 *     before anything is enqueued (B=256, gamma_max=7, V=151936 needs about
 *     1 MiB).
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for the
 *     rest of the process.  The cached address does not survive a reset of
 *     the device's primary context (cudaDeviceReset): calling this entry
 *     point after such a reset is not supported.
 *   - Every call on a device shares the one array, which each call leaves
 *     ready for the next; calls whose work may overlap on the GPU (other
 *     streams, other host threads) race on it and must be serialised by the
 *     caller, e.g. by issuing them on one stream.
 *   - Invalid per-request data is reported through out_num_accepted = -1
 *     (the error word of sv_last_error lives in the scratch array and is not
 *     exposed).
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library
 *     call is made.
 */
#define SV_NOALLOC_SCRATCH_BYTES (4u << 20)
SV_API sv_status spec_verify_noalloc(const void *target_logits, sv_dtype logits_dtype,
                                     const int32_t *draft_token_ids,
                                     const float *draft_probs,
                                     const float *uniforms_accept,
                                     const float *uniforms_sample,
                                     const float *temperature,
                                     const int32_t *draft_lens, int B, int gamma_max,
                                     int V, int32_t *out_tokens,
                                     int32_t *out_num_accepted, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
