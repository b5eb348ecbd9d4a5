/*
 * csp.h — cascade attention over a shared-prefix paged KV cache (C ABI).
 *
 * The library (libcsp_gb300.so, built for sm_103a) exposes the steps of
 * cascade attention as described on "vLLM Cascade Attention：用法、场景与原理解析"
 * (beaiera.top):
 *   - cascade_plan   : §八 Step 1-2 and §三 — the common-prefix planner and the
 *                      use-cascade decision (host only);
 *   - cascade_attn   : §一, §四 and §八 Step 5 — prefix phase (every query of the
 *                      batch, non-causal, over the shared KV pages), suffix phase
 *                      (each request, causal, over its own KV pages) and the LSE
 *                      merge, in one call;
 *   - paged_attn     : §五 and §十 — the standard (flat) path, each request over
 *                      all of its KV pages, causal;
 *   - merge_states   : §一 and §八 Step 5 (merge_attn_states) — the LSE merge of
 *                      two partial results.
 * Running-set semantics follow "fix(v1/kv_cache): resolve async KV transfer bug
 * in cascade attention #23485": the planner sees exactly the rows passed in, which
 * must be the requests that are running.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts (row-major, contiguous, no padding between rows):
 *   q        bf16  [total_q, num_q_heads, head_dim]   queries of all requests, request
 *                                                    r owning rows cu_seqlens_q[r] ..
 *                                                    cu_seqlens_q[r+1]-1
 *   k_cache, v_cache
 *            bf16  [num_blocks, block_size, num_kv_heads, head_dim]
 *   block_table int32 [num_reqs, bt_row_stride]      physical block of each logical
 *                                                    page; only the first
 *                                                    cdiv(seqused_k[r], block_size)
 *                                                    entries of row r are used (the
 *                                                    decode schedule may read entries
 *                                                    past them, within the row's
 *                                                    bt_row_stride, and ignores them)
 *   cu_seqlens_q int32 [num_reqs + 1], cu_seqlens_q[0] = 0, nondecreasing
 *   seqused_k    int32 [num_reqs]  KV length of each request, including this step's
 *                                  query tokens (queries are the last q_len positions)
 *   out      bf16  [total_q, num_q_heads, head_dim]
 *   lse      fp32  [total_q, num_q_heads]  natural log of sum_j exp(scale * q.k_j)
 * Query head h reads KV head h / (num_q_heads / num_kv_heads).  Query i of request r
 * sits at absolute position seqused_k[r] - q_len_r + i and sees keys at positions
 * <= its own (bottom-right causal alignment).
 *
 * Supported shapes: head_dim 64 or 128; block_size 16; num_q_heads a multiple of
 * num_kv_heads with a group size (num_q_heads / num_kv_heads) of 1, 2, 4, 8 or 16.
 * Anything else returns CSP_ERR_UNSUPPORTED without launching.
 *
 * Ownership: every pointer is owned by the caller.  The library allocates nothing,
 * frees nothing and keeps no pointer after a call returns.  Device pointers must
 * stay valid until the work queued on `stream` has finished.
 *
 * Asynchrony: device entry points queue kernels on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and return without synchronising.
 *
 * Errors: a negative return value means nothing was launched (argument errors), or
 * that a launch failed (CSP_ERR_CUDA, with the CUDA error kept for
 * csp_last_cuda_error()).  No C++ exception crosses the ABI.  Kernels never trap:
 * a wait inside a kernel that runs out of time writes CSP_ERR_TIMEOUT into the
 * workspace status word (see csp_workspace_status) and the kernel returns.
 *
 * Thread safety: calls may be made from several host threads at once on different
 * workspaces.  Two calls that share a workspace must be ordered on one stream.
 */
#ifndef CSP_H_
#define CSP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSP_API __attribute__((visibility("default")))
#else
#define CSP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSP_OK = 0,
  CSP_ERR_INVALID_ARG = -1,  /* null pointer, negative size, inconsistent shapes  */
  CSP_ERR_UNSUPPORTED = -2,  /* head_dim / block_size / group size not built       */
  CSP_ERR_WORKSPACE = -3,    /* workspace missing, too small or misaligned          */
  CSP_ERR_CUDA = -4,         /* a CUDA call or launch failed                        */
  CSP_ERR_TIMEOUT = -6       /* device-side: a bounded wait inside a kernel gave up */
} csp_status;

/* cascade_plan modes. */
enum {
  CSP_MODE_AUTO = 0,            /* GB300 rule: cascade when the standard path would
                                   stream >= 8192 KV tokens and cascade cuts them by
                                   >= 1.8x (fitted to a measured sweep)               */
  CSP_MODE_FORCE_CASCADE = 1,   /* use cascade whenever common_prefix_len > 0          */
  CSP_MODE_FORCE_FLAT = 2,      /* never use cascade                                   */
  CSP_MODE_PAGE_THRESHOLDS = 3  /* the pages' rule only: prefix >= 256 and batch >= 8  */
};

/* Element type of the partial results given to merge_states. */
enum { CSP_DTYPE_BF16 = 0, CSP_DTYPE_F32 = 1 };

/*
 * cascade_plan — common prefix of the running batch and the use-cascade decision.
 * Host pointers only; no device work.
 *
 * Follows §八 Step 1 (longest run, from block 0, of physical block ids shared by
 * every row), §八 Step 2 (common_prefix_len = blocks * block_size, capped to
 * min(num_computed_tokens), floored to a multiple of block_size; the cap keeps the
 * non-causal prefix phase from seeing a later token, §四), and §三 (no cascade for
 * a prefix under 256 tokens or fewer than 8 requests).  Row r takes part only with
 * its first cdiv(seq_lens[r], block_size) entries; the scan stops at the first
 * mismatch.
 *
 *   block_table          int32 [num_reqs, bt_row_stride]  host
 *   seq_lens             int32 [num_reqs]  host, KV length incl. this step's queries
 *   num_computed_tokens  int32 [num_reqs]  host, seq_lens minus this step's queries
 *   num_q_heads, num_kv_heads, head_dim   shape of the attention (cost model input)
 *   num_sms              SM count for the cost model (<= 0: 148)
 *   mode                 CSP_MODE_*
 *   common_prefix_len_out  receives the capped, floored prefix length (tokens)
 *   use_cascade_out        receives 1 to take cascade_attn, 0 for paged_attn
 * num_reqs == 0 gives 0 / 0.  Returns CSP_OK or CSP_ERR_INVALID_ARG.
 */
CSP_API int cascade_plan(const int32_t* block_table, int64_t bt_row_stride, int32_t num_reqs,
                 const int32_t* seq_lens, const int32_t* num_computed_tokens,
                 int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                 int32_t head_dim, int32_t num_sms, int32_t mode,
                 int32_t* common_prefix_len_out, int32_t* use_cascade_out);

/*
 * csp_validate_batch — optional host-side check of a batch before it is launched.
 * Host pointers only; no device work.  The kernels read the block ids they are given
 * without a bounds check (by TMA or 16-byte copies), so an id past the cache reads
 * whatever memory lies there; a caller that cannot vouch for its tables runs this on
 * the host copies first and launches only on CSP_OK.
 *
 * Checks, in this order: num_reqs >= 0, block_size > 0, num_blocks > 0; for every
 * request r: 0 <= seq_lens[r] and cdiv(seq_lens[r], block_size) <= bt_row_stride;
 * every block id a request uses (its first cdiv(seq_lens[r], block_size) entries —
 * the same entries cascade_plan scans and the kernels read) lies in [0, num_blocks);
 * if cu_seqlens_q is given: cu_seqlens_q[0] == 0 and
 * 0 <= cu_seqlens_q[r+1] - cu_seqlens_q[r] <= seq_lens[r]; common_prefix_len is a
 * multiple of block_size in [0, min_r seq_lens[r]] (0 for num_reqs == 0).
 *
 *   block_table   int32 [num_reqs, bt_row_stride]  host
 *   seq_lens      int32 [num_reqs]  host
 *   cu_seqlens_q  int32 [num_reqs + 1]  host, or NULL to skip the query checks
 *   bad_index_out NULL, or receives the flat index (r * bt_row_stride + j) of the
 *                 first out-of-range block id, or -1 when the first problem is not a
 *                 block id (and -1 on CSP_OK)
 * Returns CSP_OK or CSP_ERR_INVALID_ARG (the first problem found).
 */
CSP_API int csp_validate_batch(const int32_t* block_table, int64_t bt_row_stride,
                               int32_t num_reqs, const int32_t* seq_lens,
                               const int32_t* cu_seqlens_q, int32_t block_size,
                               int32_t num_blocks, int32_t common_prefix_len,
                               int64_t* bad_index_out);

/*
 * csp_workspace_size — bytes of device workspace that cascade_attn (with this
 * common_prefix_len) or paged_attn (common_prefix_len = 0) needs for this batch
 * shape on the current device.  All arguments are host integers, the same as the
 * attention call will get.  The workspace holds a status word, the grid barrier's
 * arrival count of the single-kernel schedule, one word per (query token, KV head) and
 * the split partial results; it must be 256-byte aligned and zero-filled before its
 * first use, and is not to be modified between calls except for zeroing it all again
 * (each call leaves its merge counters at zero and the arrival count at a multiple of
 * the device's SM count, so one workspace may serve batches of different shapes on
 * one device).  After a call reported CSP_ERR_TIMEOUT, zero the workspace again
 * before reusing it.
 * Returns CSP_OK and writes *bytes_out, or CSP_ERR_INVALID_ARG / CSP_ERR_CUDA.
 */
CSP_API int csp_workspace_size(int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                       int32_t max_seqlen_k, int32_t common_prefix_len, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, size_t* bytes_out);

/* csp_cascade_schedule results. */
enum { CSP_SCHEDULE_TWO_KERNELS = 0, CSP_SCHEDULE_SINGLE = 1, CSP_SCHEDULE_FUSED = 2 };

/*
 * csp_cascade_schedule — which kernels cascade_attn launches for a batch of this
 * shape on the current device.  Host integers, the same as the attention call will
 * get (common_prefix_len > 0).
 *   CSP_SCHEDULE_TWO_KERNELS : a prefix-phase kernel, and beside it (on the SMs it
 *                              leaves free) a paged kernel for the suffix phase that
 *                              writes its partial results; a third kernel merges
 *                              every row once both are done (any batch);
 *   CSP_SCHEDULE_SINGLE      : one cooperative kernel of one CTA per SM, for batches
 *                              where every request has at most 16 / (num_q_heads /
 *                              num_kv_heads) query tokens: some CTAs run ranges of the
 *                              prefix phase while the others stream the suffix
 *                              phase, then every CTA merges a share of the rows;
 *   CSP_SCHEDULE_FUSED       : one launch of one CTA per SM for any batch: the prefix
 *                              phase's CTAs first, then suffix CTAs on tcgen05 (up to
 *                              256 query rows of one request and KV head each); every
 *                              CTA counts itself in the row groups it covered and a
 *                              group's last contributor merges its rows.
 * Writes *schedule_out and, when prefix_splits_out is not NULL, the number of key
 * ranges the prefix phase is cut into (one workspace slot each).  Returns CSP_OK,
 * CSP_ERR_INVALID_ARG, CSP_ERR_UNSUPPORTED or CSP_ERR_CUDA.
 */
CSP_API int csp_cascade_schedule(int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                                 int32_t max_seqlen_k, int32_t common_prefix_len,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t* schedule_out, int32_t* prefix_splits_out);

/*
 * cascade_attn — cascade attention for one batch (§八 Step 5).
 *
 * Prefix phase: all total_q queries, as one sequence, attend without a causal mask
 * to KV positions [0, common_prefix_len), read through row 0 of block_table (the
 * rows share these pages; that is what the planner established).  Suffix phase:
 * request r attends causally to KV positions [common_prefix_len, seqused_k[r]),
 * read through its own row starting at page common_prefix_len / block_size.  The
 * two partial results are merged by LSE rescaling into out (bf16) and lse.
 *
 *   q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, out  device pointers,
 *                        layouts as above
 *   num_blocks           first dimension of k_cache / v_cache
 *   num_reqs, total_q    host copies of the batch size and cu_seqlens_q[num_reqs]
 *   max_seqlen_q         host: max over r of the query count of request r
 *   max_seqlen_k         host: max over r of seqused_k[r]
 *   common_prefix_len    multiple of block_size, and at most min over r of
 *                        (seqused_k[r] - q_len_r) — cascade_plan gives such a value;
 *                        0 computes the standard result
 *   softmax_scale        multiplies q.k before the softmax
 *   lse                  device pointer or NULL (not written)
 *   workspace            device, >= csp_workspace_size(...) bytes, 256-byte aligned
 *   stream               cudaStream_t
 * Results equal paged_attn's up to rounding (the pages state the two are
 * mathematically the same, §一).
 */
CSP_API int cascade_attn(const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                 const int32_t* block_table, int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                 const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                 int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t common_prefix_len,
                 int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                 float softmax_scale, void* out, float* lse, void* workspace,
                 size_t workspace_bytes, void* stream);

/*
 * cascade_attn_scheduled — cascade_attn with the schedule given by the caller instead
 * of the cost model's (for tests and tuning; results are the same up to rounding):
 *   schedule       CSP_SCHEDULE_TWO_KERNELS, CSP_SCHEDULE_FUSED, or
 *                  CSP_SCHEDULE_SINGLE where that kernel can run (a request's rows of
 *                  one KV head fit 16 and the prefix's 256-row blocks x KV heads fit
 *                  the SMs; else CSP_ERR_UNSUPPORTED)
 *   prefix_ranges  > 0: the number of prefix key ranges of the single kernel (capped at
 *                  15, the prefix's 64-key tiles and the SMs' room) or of the
 *                  two-kernel schedule when a request and KV head have at most 16
 *                  query rows (capped at 16 and the prefix's 64-key tiles); 0: the
 *                  cost model's
 * common_prefix_len must be > 0.  Other arguments, the workspace (csp_workspace_size
 * covers every schedule and number of ranges) and the errors are cascade_attn's;
 * CSP_ERR_INVALID_ARG for an unknown schedule or a negative prefix_ranges.
 */
CSP_API int cascade_attn_scheduled(const void* q, const void* k_cache, const void* v_cache,
                                   int32_t num_blocks, const int32_t* block_table,
                                   int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                                   const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                                   int32_t max_seqlen_q, int32_t max_seqlen_k,
                                   int32_t common_prefix_len, int32_t block_size,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   float softmax_scale, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, void* stream, int32_t schedule,
                                   int32_t prefix_ranges);

/*
 * cascade_attn_timed — cascade_attn plus four CUDA events recorded on `stream`
 * between its kernels, for timing each phase.  Two-kernel schedule:
 * phase_events[0] before the prefix-phase kernel, [1] after it, [2] after the
 * suffix-phase kernel (whose CTAs finish the LSE merge, or which is followed by the
 * merge kernel: see csp_cascade_schedule), [3] at the end of the call (after the merge
 * kernel where there is one, else the same point as [2]); with events between them,
 * the kernels run one after
 * the other instead of overlapping, so the per-phase times add up to more than a
 * cascade_attn call takes; with common_prefix_len == 0, events [0] and [1] mark the
 * same point.  Single-kernel schedule (csp_cascade_schedule): [0] before the kernel,
 * [1], [2] and [3] after it.  phase_events is a host array of four cudaEvent_t
 * created by the caller (with timing enabled).  Arguments and results are otherwise
 * those of cascade_attn.
 */
CSP_API int cascade_attn_timed(const void* q, const void* k_cache, const void* v_cache,
                               int32_t num_blocks, const int32_t* block_table,
                               int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                               const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                               int32_t max_seqlen_q, int32_t max_seqlen_k,
                               int32_t common_prefix_len, int32_t block_size,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               float softmax_scale, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream,
                               void* const* phase_events);

/*
 * cascade_attn_noalloc — cascade_attn for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment convenience of this library.
 *
 * Who needs it: code that runs attention where cudaMalloc is off limits, such as an
 * engine that hands out all device memory from its own pool up front, a plugin
 * inside a framework that owns every allocation, or a latency-critical loop where an
 * allocation could synchronise the device.  Such a caller passes inputs and outputs
 * exactly as for cascade_attn, but no workspace: the library uses a fixed 16 MiB
 * array of its own device memory instead (reserved on each GPU where the library's
 * device code is loaded, and held until the process exits).  Nothing is allocated
 * or freed by this call.
 *
 * The first call on a device looks up that array's device address (once per device
 * and context, with the device current); make that first call before any stream
 * capture.  A context that is destroyed and created again (cudaDeviceReset) gets a new
 * array, whose address the next call looks up the same way.  Every
 * call on a device shares the one array: calls that can run at the same time on the
 * GPU (different streams, no ordering between them) race and corrupt each other's
 * results; order them on one stream.  The array keeps the previous call's contents;
 * each call clears the status word at its start itself.  A batch whose workspace
 * (csp_workspace_size) exceeds 16 MiB is rejected with CSP_ERR_WORKSPACE before
 * anything is launched.  A bounded wait inside the kernels that gives up writes
 * CSP_ERR_TIMEOUT into the array's status word, as for a caller's workspace: read it
 * with csp_noalloc_status after the call and before the next one (each call clears
 * it).  Other arguments, layouts and errors: as for cascade_attn.
 */
CSP_API int cascade_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 int32_t num_blocks, const int32_t* block_table,
                                 int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                                 const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                                 int32_t max_seqlen_q, int32_t max_seqlen_k,
                                 int32_t common_prefix_len, int32_t block_size,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 float softmax_scale, void* out, float* lse, void* stream);

/*
 * csp_noalloc_status — the status word of the array cascade_attn_noalloc uses on the
 * current device, copied to the host (a blocking copy on `stream`; order it after the
 * call it checks).  0: the last call's kernels reported no problem; CSP_ERR_TIMEOUT: a
 * bounded wait gave up and that call's out/lse are not valid.  Writes *status_out.
 * No counterpart on the pages (it belongs to cascade_attn_noalloc).  Allocates
 * nothing.
 */
CSP_API int csp_noalloc_status(void* stream, int32_t* status_out);

/*
 * paged_attn — the standard path (§五, §十): request r attends causally to all of
 * its KV positions [0, seqused_k[r]) through its own block_table row.  Arguments
 * as for cascade_attn, without common_prefix_len.
 */
CSP_API int paged_attn(const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
               const int32_t* block_table, int64_t bt_row_stride, const int32_t* cu_seqlens_q,
               const int32_t* seqused_k, int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
               int32_t max_seqlen_k, int32_t block_size, int32_t num_q_heads,
               int32_t num_kv_heads, int32_t head_dim, float softmax_scale, void* out,
               float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * merge_states — LSE merge of two partial attention results over disjoint key sets
 * (merge_attn_states, §一 and §八 Step 5):
 *   m = max(l1, l2); out = (e^(l1-m) o1 + e^(l2-m) o2) / (e^(l1-m) + e^(l2-m));
 *   out_lse = m + ln(e^(l1-m) + e^(l2-m)).
 * Rows where both lse are -inf give out = 0 and out_lse = -inf.
 *
 *   out          device bf16 [num_tokens, num_heads, head_dim]
 *   out_lse      device fp32 [num_tokens, num_heads] or NULL
 *   prefix_out, suffix_out   device, [num_tokens, num_heads, head_dim] of partial_dtype
 *   prefix_lse, suffix_lse   device fp32 [num_tokens, num_heads], natural log
 *   partial_dtype            CSP_DTYPE_BF16 or CSP_DTYPE_F32
 * head_dim must be a multiple of 8 and at most 512.
 */
CSP_API int merge_states(void* out, float* out_lse, const void* prefix_out, const float* prefix_lse,
                 const void* suffix_out, const float* suffix_lse, int32_t num_tokens,
                 int32_t num_heads, int32_t head_dim, int32_t partial_dtype, void* stream);

/*
 * cascade_plan_device — the common-prefix planner as one small kernel on `stream`, for
 * steps captured in a CUDA graph.  §十一: cascade does not fit a full CUDA graph when
 * the use-cascade decision is taken per batch on the host and the number of kernel
 * calls follows it; §七: FlashInfer splits a plan step from a run step so that the run
 * can be captured.  Here the plan reads the batch where it already is (device memory)
 * and leaves its result there for cascade_attn_device_plan, so a step is the same
 * fixed launches whatever the batch.  The arithmetic is cascade_plan's (§八 Step 1-2,
 * §三, and the same modes), with the same results.
 *
 *   block_table          device int32 [num_reqs, bt_row_stride]
 *   seq_lens             device int32 [num_reqs]
 *   num_computed_tokens  device int32 [num_reqs]
 *   plan_out             device int32 [4]: [0] the prefix length for the attention call
 *                        (common_prefix_len when cascade is taken, else 0), [1]
 *                        use_cascade, [2] common_prefix_len, [3] status (CSP_OK, or
 *                        CSP_ERR_INVALID_ARG for lengths cascade_plan would refuse, with
 *                        [0..2] = 0)
 * Asynchronous; no device-to-host copy.  Returns CSP_OK, CSP_ERR_INVALID_ARG (nothing
 * launched) or CSP_ERR_CUDA.
 */
CSP_API int cascade_plan_device(const int32_t* block_table, int64_t bt_row_stride,
                                int32_t num_reqs, const int32_t* seq_lens,
                                const int32_t* num_computed_tokens, int32_t block_size,
                                int32_t mode, int32_t* plan_out, void* stream);

/*
 * cascade_attn_device_plan — cascade_attn with the prefix length read from device
 * memory (plan[0], as cascade_plan_device leaves it) when the kernel runs, so that the
 * pair can be captured in a CUDA graph once and replayed for every batch that fits the
 * launch plan.  The launch plan (grid, prefix key ranges, workspace partition) is made
 * on the host for common_prefix_len_bound, a multiple of block_size at least as large
 * as any plan[0] the launch will read (plan[0] is clamped to it); plan[0] = 0 computes
 * the standard path.  Only the single-kernel schedule reads its prefix length from
 * device memory: batches it does not take (more than 16 packed rows per request and
 * KV head, more than 8 KV heads, or too many 256-row blocks) and a bound of 0 return
 * CSP_ERR_UNSUPPORTED with nothing launched.  Size the workspace with
 * csp_workspace_size for common_prefix_len_bound.  Other arguments, layouts and
 * errors: as for cascade_attn.
 */
CSP_API int cascade_attn_device_plan(const void* q, const void* k_cache, const void* v_cache,
                                     int32_t num_blocks, const int32_t* block_table,
                                     int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                                     const int32_t* seqused_k, int32_t num_reqs,
                                     int32_t total_q, int32_t max_seqlen_q,
                                     int32_t max_seqlen_k, const int32_t* plan,
                                     int32_t common_prefix_len_bound, int32_t block_size,
                                     int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, float softmax_scale, void* out,
                                     float* lse, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * csp_apply_sinks — attention sinks (§九 "Attention Sinks": every backend takes an
 * optional `sinks` argument).  Each query head h has one sink logit s_h (natural log,
 * not multiplied by the softmax scale) that joins the softmax of every row of head h
 * as one more key whose value row is zero.  Applied to a finished result of
 * cascade_attn or paged_attn (its out and natural-log lse) as the LSE merge (§一,
 * merge_attn_states) with an empty partial whose lse is s_h:
 *     lse' = ln(e^lse + e^s_h),   out' = out * e^(lse - lse')
 * so the step is exact up to one more bf16 rounding of out.  s_h = -inf leaves a row
 * unchanged; a row with no key (lse = -inf) keeps out = 0 and gets lse' = s_h.
 *
 *   out     device bf16 [num_tokens, num_heads, head_dim], 16-byte aligned, in place
 *   lse     device fp32 [num_tokens, num_heads], natural log, in place (required)
 *   sinks   device fp32 [num_heads]
 *   head_dim  a multiple of 8 with head_dim / 8 dividing 32 (8 ... 256)
 * Asynchronous on `stream`; order it after the attention call that wrote out and lse.
 * Returns CSP_OK, CSP_ERR_INVALID_ARG (nothing launched) or CSP_ERR_CUDA.
 */
CSP_API int csp_apply_sinks(void* out, float* lse, const float* sinks, int32_t num_tokens,
                            int32_t num_heads, int32_t head_dim, void* stream);

/*
 * FP8 KV cache.  §六: FlashInfer's cascade wrapper is switched off for a KV cache
 * stored in FP8.  These entry points take K and V caches of E4M3 bytes (OCP FP8 E4M3,
 * "e4m3fn": bias 7, no infinities, S.1111.111 = NaN) in the usual layout
 * [num_blocks, block_size, num_kv_heads, head_dim], each with one scale per tensor:
 * an element's value is decode(byte) * k_scale (or * v_scale), and the result is the
 * attention over those values.  The kernels widen the bytes to f16 (exact: every
 * E4M3 value is an f16 value) and compute in f16 with fp32 accumulation: the queries
 * are converted to f16 first (exact for bf16 values in f16's normal range, |q| in
 * [2^-14, 65504]; rounded to f16's subnormal grid below it), k_scale is folded into
 * the softmax scale and v_scale into the normalised output.  Half the KV bytes of a
 * bf16 cache are read.
 *
 * csp_workspace_size_fp8kv — workspace bytes of cascade_attn_fp8kv (common_prefix_len
 * > 0) or paged_attn_fp8kv (0): the plan's partials plus an f16 copy of q.  Errors as
 * for csp_workspace_size.
 */
CSP_API int csp_workspace_size_fp8kv(int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                                     int32_t max_seqlen_k, int32_t common_prefix_len,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                     size_t* bytes_out);

/*
 * cascade_attn_fp8kv / paged_attn_fp8kv — cascade_attn and paged_attn over an E4M3 KV
 * cache (k_cache, v_cache: device uint8, 16-byte aligned) with scales k_scale, v_scale
 * (finite, > 0; else CSP_ERR_INVALID_ARG).  They run the two-kernel schedule (the
 * prefix kernel and the paged kernels with the tiles widened in shared memory) and
 * need csp_workspace_size_fp8kv bytes of workspace (else CSP_ERR_WORKSPACE).  Other
 * arguments, layouts and errors: as for cascade_attn and paged_attn.
 */
CSP_API int cascade_attn_fp8kv(const void* q, const void* k_cache, const void* v_cache,
                               int32_t num_blocks, const int32_t* block_table,
                               int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                               const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                               int32_t max_seqlen_q, int32_t max_seqlen_k,
                               int32_t common_prefix_len, int32_t block_size,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               float softmax_scale, float k_scale, float v_scale, void* out,
                               float* lse, void* workspace, size_t workspace_bytes,
                               void* stream);
CSP_API int paged_attn_fp8kv(const void* q, const void* k_cache, const void* v_cache,
                             int32_t num_blocks, const int32_t* block_table,
                             int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                             const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                             int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t block_size,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             float softmax_scale, float k_scale, float v_scale, void* out,
                             float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Multi-level cascade.  §七: FlashInfer's cascade runs any number of levels
 * (num_levels) where vLLM's runs two.  The levels form a prefix tree over consecutive
 * requests: a segment (level, r_lo, r_hi, k_lo, k_hi) is a run of at least two
 * consecutive requests [r_lo, r_hi) that share the blocks of keys [k_lo, k_hi), the
 * keys right after those of the level - 1 segment that holds them (level 0: from key
 * 0).  Each segment is found as §八 Step 1-2 finds the common prefix, within its own
 * requests and from k_lo: the longest run of shared block ids, capped to the
 * segment's minimum num_computed_tokens and floored to block_size.  A request's suffix
 * starts at the end of the deepest segment that holds it (0 when none does).  A batch
 * of two families of requests over one system prompt (a shared document per family)
 * is the three-level case: the system prompt at level 0, each family's document at
 * level 1, each request's own tokens in its suffix.
 *
 * cascade_plan_levels — the planner (host only).  Walks the prefix tree depth first,
 * at most max_levels deep, and writes at most max_segments segments as 7 int32 each:
 * level, r_lo, r_hi, k_lo, k_hi and the segment's query rows tok_lo, tok_hi (its
 * requests' query tokens, q_len_r = seq_lens[r] - num_computed_tokens[r]); writes
 * *num_segments_out and suffix_start_out[num_reqs] (host).  Block table and lengths:
 * host arrays as for cascade_plan.  Returns CSP_OK, CSP_ERR_INVALID_ARG (lengths
 * cascade_plan would refuse, max_levels outside 1..8) or CSP_ERR_UNSUPPORTED (more
 * than max_segments segments).
 */
CSP_API int cascade_plan_levels(const int32_t* block_table, int64_t bt_row_stride,
                                int32_t num_reqs, const int32_t* seq_lens,
                                const int32_t* num_computed_tokens, int32_t block_size,
                                int32_t max_levels, int32_t max_segments,
                                int32_t* segments_out, int32_t* num_segments_out,
                                int32_t* suffix_start_out);

/*
 * csp_workspace_size_levels — workspace bytes cascade_attn_levels needs for these
 * segments (host array, as cascade_plan_levels writes them) and a longest suffix of
 * max_suffix_len keys (max over r of seqused_k[r] - suffix_start[r]).  Returns
 * CSP_OK, CSP_ERR_INVALID_ARG, CSP_ERR_UNSUPPORTED (the shapes cascade_attn refuses;
 * more than 24 prefix slots: the levels' largest key-range splits added up) or
 * CSP_ERR_CUDA (no device to size the grid for).
 */
CSP_API int csp_workspace_size_levels(int32_t num_reqs, int32_t total_q, int32_t max_seqlen_q,
                                      int32_t max_seqlen_k, const int32_t* segments,
                                      int32_t num_segments, int32_t max_suffix_len,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, size_t* bytes_out);

/*
 * cascade_attn_levels — attention through a multi-level cascade: every segment's
 * query rows over its shared keys (non-causal: the keys lie within every one of its
 * requests' computed tokens), each request's suffix keys [suffix_start[r],
 * seqused_k[r]) causal, and the LSE merge of all of them; the result equals the
 * standard path's up to rounding.  segments: host int32 [num_segments][7] as
 * cascade_plan_levels writes them (the key ranges of the segments that hold a request
 * must follow one another from key 0 to its suffix start; two segments of one level
 * hold no request in common; each within every one of its requests' computed tokens);
 * suffix_start: device int32 [num_reqs]; max_suffix_len as for
 * csp_workspace_size_levels.  Segments of one level write that level's slots of the
 * workspace; a row no segment of a level holds has an empty slot there (lse -inf).
 * Other arguments, layouts and errors: as for cascade_attn; segments that break the
 * host-checkable rules above return CSP_ERR_INVALID_ARG with nothing launched.
 */
CSP_API int cascade_attn_levels(const void* q, const void* k_cache, const void* v_cache,
                                int32_t num_blocks, const int32_t* block_table,
                                int64_t bt_row_stride, const int32_t* cu_seqlens_q,
                                const int32_t* seqused_k, int32_t num_reqs, int32_t total_q,
                                int32_t max_seqlen_q, int32_t max_seqlen_k,
                                const int32_t* segments, int32_t num_segments,
                                const int32_t* suffix_start, int32_t max_suffix_len,
                                int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, float softmax_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * cascade_step_host — one whole step from host buffers: copies the step's q, block
 * table, cu_seqlens_q and seq_lens to the device, plans on the host (cascade_plan with
 * `mode`; the standard path when it declines cascade), runs the attention call, copies
 * out and lse back and waits for them (a stream synchronisation), so out and lse hold
 * the result when it returns.  For a user whose batch lives in host memory; pinned
 * (page-locked) host buffers let the copies run asynchronously.
 *
 *   q                    host bf16 [total_q, num_q_heads, head_dim]
 *   block_table          host int32 [num_reqs, bt_row_stride]
 *   cu_seqlens_q         host int32 [num_reqs + 1]
 *   seq_lens             host int32 [num_reqs]
 *   num_computed_tokens  host int32 [num_reqs] (the planner's cap)
 *   k_cache, v_cache     device, as for cascade_attn (resident, as in serving)
 *   out, lse             host bf16 [total_q, num_q_heads, head_dim], fp32 [total_q,
 *                        num_q_heads] (natural log), written
 *   device_scratch       device, 256-byte aligned, csp_step_scratch_size bytes for the
 *                        prefix length the planner returns (0 and that length cover both
 *                        paths), zero-filled before its first use: it holds the
 *                        attention call's workspace at its start, then the step's device
 *                        copies
 *   common_prefix_len_out  the prefix length used (0: the standard path), or NULL
 * Returns CSP_OK, the planner's or cascade_attn's errors (nothing launched on an
 * argument error), CSP_ERR_WORKSPACE, or CSP_ERR_CUDA.
 *
 * csp_step_scratch_size — device_scratch bytes for such a step with a given prefix
 * length (host arrays as above).
 */
CSP_API int csp_step_scratch_size(int32_t num_reqs, int32_t total_q, const int32_t* cu_seqlens_q,
                                  const int32_t* seq_lens, int64_t bt_row_stride,
                                  int32_t common_prefix_len, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, size_t* bytes_out);
CSP_API int cascade_step_host(const void* q, const int32_t* block_table, int64_t bt_row_stride,
                              const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                              const int32_t* num_computed_tokens, int32_t num_reqs,
                              int32_t total_q, const void* k_cache, const void* v_cache,
                              int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, float softmax_scale,
                              int32_t mode, void* out, float* lse, void* device_scratch,
                              size_t scratch_bytes, void* stream,
                              int32_t* common_prefix_len_out);

/*
 * csp_workspace_status — copies the workspace status word to the host (a blocking
 * copy on `stream`).  0 means no kernel reported a problem since the workspace was
 * zero-filled; CSP_ERR_TIMEOUT means a bounded wait gave up.  Writes *status_out.
 */
CSP_API int csp_workspace_status(const void* workspace, void* stream, int32_t* status_out);

/* Human-readable name of a csp_status value (static string). */
CSP_API const char* csp_status_string(int status);

/* The CUDA error code behind the last CSP_ERR_CUDA returned on this host thread. */
CSP_API int csp_last_cuda_error(void);

/* ABI version: (major << 16) | minor. */
CSP_API int csp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSP_H_ */
