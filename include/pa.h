/*
 * pa.h -- C ABI of libpa: paged-KV GQA decode attention with a
 * context-proportional split-KV work plan, for NVIDIA GB300 (sm_103a).
 *
 * The operation (sources are web pages, cited by title and section):
 *
 *   [ATOM-2366] ROCm/ATOM pull 2366, "[MiniMax-M3] Route the paged decode to
 *     aiter's FlyDSL kernel with work planner".  Section 1 (Motivation): a
 *     planner hands each request a partition count proportional to its real
 *     context length.  Section 3 (Design): the work budget is 2 x CU, the
 *     partition ceiling 256; the plan depends on context_lens only, is built
 *     once per forward, refreshed in place (no allocation, no device-to-host
 *     copy) so it can be captured in a CUDA graph.  Section 5, "Planner drift
 *     at the real ceiling": capacity = min(batch x max_partitions,
 *     max(batch, 2 x CU / kv_heads)).  Review item 2: the plan stores per-task
 *     begin/end tiles plus seq_ctx (word 3 of each 4-word task).  Review item
 *     5: the capability gate (dtypes, block size, head_dim, int32 tables,
 *     q heads divisible by kv heads, out shaped and typed like q).
 *   [ATOM-2514] ROCm/ATOM pull 2514, "Fix(attention): adapt the FlyDSL paged
 *     decode to aiter #5809 (explicit work plans)".  Motivation/Design: every
 *     decode call takes an explicit plan with the default 2 x CU budget; more
 *     than 4096 sequences is outside the planner's domain.
 *   [RDNA-29] opengfx1030/vllm-rdna pull 29 (mixed and MTP-verify batches),
 *     Change section 1 "Kernel: per-token causal decode": with cu_query_lens a
 *     request owns L = cu[r+1]-cu[r] consecutive query rows; its token i
 *     attends to the first S - (L - 1 - i) keys; rows past cu[num_seqs] and
 *     rows of zero-length requests come out as zeros; without cu_query_lens
 *     row r is request r's single token.
 *
 * For query row t of request r (token i), q head hq and kv head h = hq / G
 * (G = Hq / Hkv), with K_t = S_r - (L_r - 1 - i) visible keys:
 *     out[t, hq, :] = sum_j softmax_j(scale * <q[t,hq], k_j>) * v_j,  j < K_t,
 * k_j / v_j the j-th key/value row of request r in kv head h, gathered through
 * block_tables.  fp8 caches hold OCP float8 e4m3fn codes; a code c means
 * e4m3fn(c) * k_scale (keys) or * v_scale (values).
 *
 * Data layouts (all row-major, contiguous, device memory unless stated):
 *   q, out          [num_tokens, Hq, D]          bf16 or fp16; out has q's dtype
 *   k_cache,v_cache [num_blocks, Hkv, block_size, D]  bf16, fp16 or e4m3fn bytes
 *                   (pa_decode_ex also takes k_cache as PA_K_GROUPED:
 *                   [num_blocks, Hkv, D/16, block_size, 16])
 *   block_tables    int32 [num_seqs, max_blocks_per_seq]; entry b of row r is
 *                   the physical block holding keys [b*bs, (b+1)*bs) of r
 *   context_lens    int32 [num_seqs]  KV length of each request (query tokens
 *                   included)
 *   cu_query_lens   int32 [num_seqs + 1] or NULL; nondecreasing, cu[0] == 0
 *
 * Work plan (device memory owned by the plan):
 *   work_info   int32 [capacity][4] = (seq, tile_begin, tile_end, seq_ctx);
 *               seq = -1 marks an unused slot.  A task covers keys
 *               [tile_begin*256, min(tile_end*256, seq_ctx)).
 *   reduce_info int32 [num_seqs][2] = (first_slot, num_parts); slots are
 *               request-major, first_slot is the running sum of num_parts.
 *   Rule (integer, int64 intermediates), with n_act the requests that have
 *   S > 0 and at least one query row, and T = 256 tokens:
 *     capacity C = min(n * P, max(n, ceil(W / Hkv)))
 *     PROPORTIONAL: p_r = min(P, ceil(S_r/T), 1 + floor((C - n_act) * S_r / sum S))
 *     UNIFORM:      p_r = min(P, ceil(S_r/T), floor(C / n_act))
 *     inactive requests: p_r = 0.  Part j of request r covers tiles
 *     [floor(j*nt/p), floor((j+1)*nt/p)), nt = ceil(S_r/T).
 *   The proportional rule's integer form (reserve one partition per active
 *   request, share the rest in proportion to S with floor rounding) and the
 *   uniform comparator are this library's reading of the pages, which give no
 *   closed integer form for either.
 *
 * Streams, ownership, capture: every call that takes a stream enqueues its
 * work on that stream (a cudaStream_t passed as void*; NULL = legacy default
 * stream) and returns without synchronising, unless stated.  The caller owns
 * every tensor.  A plan owns its device buffers, allocated only by
 * pa_plan_build and released by pa_plan_destroy; pa_plan_refresh and
 * pa_decode never allocate and never wait on the host, so both may be
 * captured in a CUDA graph.  The first launch of each kernel shape on a device
 * sets that kernel's shared-memory limit and reads its occupancy there (host
 * calls, no stream work; kept per device ordinal, safe from several threads).
 * One plan may be in flight on one stream at a time
 * (its partial-result scratch is per plan).  pa_plan_refresh must run after
 * every change of context_lens or cu_query_lens and before the pa_decode
 * calls that use it; pa_decode detects a plan refreshed from other lengths and
 * reports it through the device error word (PA_DEVERR_STALE_PLAN) rather than
 * computing over the wrong key ranges.
 *
 * Errors: every function returns PA_OK or a negative PA_ERR_* status; nothing
 * aborts, throws across the ABI, or falls back to another implementation.
 * Problems only visible on the device (bad block-table entries, a stale plan,
 * lengths beyond what the plan was built for) set bits in a sticky per-plan
 * error word, read with pa_plan_read_errors.
 */
#ifndef PA_H_
#define PA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1,   /* null pointer, negative size, misaligned pointer, bad code */
  PA_ERR_UNSUPPORTED = -2,   /* outside the supported domain (dtype, D, block size, ...) */
  PA_ERR_PLAN_MISMATCH = -3, /* call disagrees with the plan (shape, never refreshed, ...) */
  PA_ERR_CUDA = -4,          /* a CUDA runtime/driver call failed (no device, launch error) */
  PA_ERR_OOM = -5            /* device allocation failed in pa_plan_build */
};

/* Element types. */
enum pa_dtype { PA_BF16 = 0, PA_FP16 = 1, PA_FP8_E4M3 = 2 };

/* K cache layouts (pa_decode_ex).  PA_K_ROWS: [num_blocks, Hkv, block_size, D].
 * PA_K_GROUPED: the 5-D [num_blocks, Hkv, D/16, block_size, 16] that the
 * capability gate of [ATOM-2366] (review items 5 and 12) checks the key cache
 * against -- the head dim cut into 16-element groups, each group's block_size
 * rows contiguous.  V is [num_blocks, Hkv, block_size, D] in both. */
enum pa_k_layout { PA_K_ROWS = 0, PA_K_GROUPED = 1 };

/* Plan kinds: the context-proportional plan, and the uniform comparator. */
enum pa_plan_kind { PA_PLAN_PROPORTIONAL = 0, PA_PLAN_UNIFORM = 1 };

/* Sticky device error bits. */
#define PA_DEVERR_STALE_PLAN 0x1u    /* lengths differ from those of the last refresh */
#define PA_DEVERR_BAD_PAGE 0x2u      /* a needed block-table entry is outside [0, num_blocks)
                                        or past max_blocks_per_seq; its keys read as zeros */
#define PA_DEVERR_PLAN_OVERFLOW 0x4u /* refresh saw a query length above max_query_len, more
                                        than max_tokens rows, or a malformed cu_query_lens;
                                        the plan was emptied (every output row becomes 0) */
#define PA_DEVERR_TIMEOUT 0x8u       /* a bounded wait inside a kernel gave up */

#define PA_TILE_TOKENS 256          /* partition tile, in tokens */
#define PA_DEFAULT_MAX_PARTITIONS 256
#define PA_MAX_SEQS 4096

typedef struct pa_plan pa_plan; /* opaque */

/* Creates a plan for batches of exactly num_seqs requests, num_kv_heads kv
 * heads and num_q_heads query heads (in that order) on device `device` and
 * allocates its device buffers: work_info, reduce_info, the per-request
 * snapshot of query lengths, the error word, and fp32 partial-result scratch
 * sized for at most max_query_len query rows per request and max_tokens rows
 * per call.  max_partitions <= 0 selects 256; budget <= 0 selects
 * 2 x multiProcessorCount of the device ([ATOM-2514] Design, "default
 * budget").  kind is a pa_plan_kind.  The plan is unusable by pa_decode until
 * the first pa_plan_refresh.  Supported: 1 <= num_seqs <= 4096, Hq % Hkv == 0,
 * head_dim 64 or a multiple of 128 up to 1024 (the [ATOM-2366] capability
 * gate, review item 5).  Returns PA_ERR_OOM / PA_ERR_CUDA on device
 * failures (nothing is leaked), PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED on bad
 * parameters.  On success *plan owns the buffers until pa_plan_destroy. */
int pa_plan_build(pa_plan** plan, int device, int num_seqs, int num_kv_heads, int num_q_heads,
                  int head_dim, int max_query_len, int max_tokens, int max_partitions, int budget,
                  int kind);

/* Recomputes the plan in place from the live device arrays context_lens
 * [num_seqs] and cu_query_lens [num_seqs + 1] (NULL: one query row per
 * request), on `stream`: one kernel, no allocation, no host synchronisation
 * ([ATOM-2366] section 3, plan lifetime vs cudagraph).  Whether cu_query_lens
 * was given is remembered: pa_decode must be called the same way. */
int pa_plan_refresh(pa_plan* plan, const int32_t* context_lens, const int32_t* cu_query_lens,
                    void* stream);

/* Paged decode over the plan's tasks, then an LSE-weighted merge of each
 * request's partial results ([ATOM-2366] sections 3 and 6 item 5: split
 * attention tile, then the partial-softmax reduce) -- inside the split kernel
 * or by a second kernel, see pa_plan_set_fused_merge.  Arguments follow the
 * layouts above; num_q_heads, head_dim, num_kv_heads and num_seqs must equal
 * the plan's.  q_dtype is PA_BF16 or PA_FP16; kv_dtype is PA_BF16 (q bf16),
 * PA_FP16 (q fp16) or PA_FP8_E4M3 (q bf16 or fp16; the dot products then run
 * on fp16 values, so |q| must stay below 65504).  k_scale / v_scale apply to
 * fp8 caches only and must be finite.  block_size in {16, 64, 128};
 * num_blocks * num_kv_heads * block_size < 2^31.  Without cu_query_lens
 * num_tokens == num_seqs; with it, num_tokens >= 1 and rows past
 * cu[num_seqs] are graph padding (written as zeros).  q, out, k_cache and
 * v_cache must be 16-byte aligned.  Every output row is written.  Enqueues
 * one kernel (fused merge) or two on `stream`; returns without waiting. */
int pa_decode(pa_plan* plan, const void* q, int q_dtype, int num_tokens, int num_q_heads,
              int head_dim, const void* k_cache, const void* v_cache, int kv_dtype, float k_scale,
              float v_scale, int num_blocks, int num_kv_heads, int block_size,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              const int32_t* cu_query_lens, int num_seqs, float scale, void* out, void* stream);

/* Sliding window ("vllm-rdna pull 29", Change 1: the window applies per
 * token; the aiter pa_decode signature the pages quote carries
 * sliding_window): with sliding_window = W > 0, query token i, whose causal
 * range is keys [0, K_i), attends only to [max(0, K_i - W), K_i); 0 (the
 * default) turns the window off.  A plan property: it takes effect at the
 * next pa_plan_refresh, which then sizes each request by the keys its tokens
 * read (from the tile holding the first token's first visible key; tile
 * indices in work_info stay absolute), and every pa_decode uses the window of
 * the plan's last refresh.  PA_ERR_INVALID_ARG for W < 0. */
int pa_plan_set_window(pa_plan* plan, int sliding_window);

/* The element type of the caches the plan's pa_decode calls will read (a
 * pa_dtype: PA_BF16 by default, PA_FP16 or PA_FP8_E4M3).  No counterpart in
 * the pages: it tells the planner how many CTAs of the decode kernel one SM
 * holds (an fp8 stage is half the size of a 16-bit one), so that when the
 * plan's CTAs (capacity x num_kv_heads) are more than the GPU runs at once,
 * the refresh cuts the tasks into pieces (at least two 256-key tiles, at most
 * four per task) that the CTAs of the first wave share, instead of leaving a
 * second, partly empty wave of whole tasks.  work_info and reduce_info do not
 * change; a pa_decode over another cache type stays correct.  Takes effect at
 * the next pa_plan_refresh.  PA_ERR_INVALID_ARG for another value. */
int pa_plan_set_kv_dtype(pa_plan* plan, int kv_dtype);

/* Where pa_decode merges the partial results of requests split into several
 * pieces ([ATOM-2366] section 6 item 5 and review item 7: the partial-softmax
 * reduce after the split attention tiles, which the pages measured ~14%
 * dearer as a separate pass).  enable = 1: the split kernel merges them itself
 * -- the CTA that finishes the last piece of a group of up to 8 takes the
 * group's last ticket (an atomic count, no waiting) and merges the group, up a
 * tree until the request's output rows are written -- and pa_decode launches
 * one kernel; enable = 0: a separate merge kernel runs after the split kernel.
 * The fused merge is possible for plans whose requests' query rows
 * (max_query_len x the GQA group) fit one work item of the split kernel (at
 * most 32 rows) and whose head_dim is at most 256; every other plan keeps the
 * merge kernel, where a request's many query rows are better spread over many
 * CTAs.  The default is 0 for every plan: on GB300 the merge kernel, chained
 * to the split kernel by programmatic dependent launch, measured faster per
 * decode call on every batch tried -- 1.2-8 us on one-row decode (the ticket
 * round trip after each piece stalls that CTA's pipeline), 5-9 us on 2-4-token
 * verify rows and 21 us on 3-token verify at head dim 256 (the CTA that takes
 * a request's last ticket merges all L x G rows of its pieces with a few
 * warps, where the merge kernel spreads them over many CTAs).
 * PA_ERR_UNSUPPORTED for enable = 1 on such a plan, PA_ERR_INVALID_ARG for
 * another value.  Takes effect at the next pa_decode.  No counterpart in the
 * pages beyond the cost they measured. */
int pa_plan_set_fused_merge(pa_plan* plan, int enable);

/* Whether the plan's pa_decode calls merge in the split kernel (1) or in a
 * separate merge kernel (0). */
int pa_plan_get_fused_merge(const pa_plan* plan, int* enabled);

/* Limit of the decode kernel's bounded waits, for the plan's later pa_decode
 * calls: a wait on a pipeline stage that has not completed after wait_limit_ns
 * nanoseconds gives up, raises PA_DEVERR_TIMEOUT in the plan's error word and
 * abandons that CTA's remaining work (its output rows are then meaningless);
 * the kernel still returns and the context stays usable.  0 restores the
 * default of 4 s; otherwise at least 10 us (PA_ERR_INVALID_ARG below that or
 * for a negative value).  No counterpart in the pages. */
int pa_plan_set_wait_limit(pa_plan* plan, long long wait_limit_ns);

/* Test hook for the timeout path: with stage >= 0, the producer of every CTA
 * of the plan's later pa_decode calls leaves its pipeline stage number `stage`
 * (counted from 0 across the CTA's work items) neither copied nor armed, so
 * every wait on it runs out after the wait limit and PA_DEVERR_TIMEOUT is
 * raised; -1 (the default) turns it off.  The results of such a call are
 * meaningless.  PA_ERR_INVALID_ARG below -1.  No counterpart in the pages. */
int pa_plan_skip_stage_for_test(pa_plan* plan, int stage);

/* pa_decode with attention sinks and a choice of K layout.  sinks (named in
 * the same aiter signature) is NULL or a device array of num_q_heads fp32
 * logits, in the units of scale * q.k, each joining its head's softmax
 * denominator only: out = sum_j e^(s_j) v_j / (sum_j e^(s_j) + e^(sink)).  A
 * row with no visible key is still 0.  k_layout is a pa_k_layout (the same
 * bytes of keys either way; results are identical up to summation order);
 * PA_ERR_UNSUPPORTED for another value.  Everything else is as pa_decode
 * (which is this call with sinks = NULL and k_layout = PA_K_ROWS). */
int pa_decode_ex(pa_plan* plan, const void* q, int q_dtype, int num_tokens, int num_q_heads,
                 int head_dim, const void* k_cache, const void* v_cache, int kv_dtype,
                 float k_scale, float v_scale, int num_blocks, int num_kv_heads, int block_size,
                 const int32_t* block_tables, int max_blocks_per_seq,
                 const int32_t* context_lens, const int32_t* cu_query_lens, int num_seqs,
                 float scale, const float* sinks, int k_layout, void* out, void* stream);

/* Sparse top-k block selection, for the sparse decode of [ATOM-2366] section 3
 * (the sparse call sites read a fixed top-k window) and [ATOM-2514] Design
 * ("Once-per-step sparse refresh": the local tail block is always selected, so
 * a request's selected length depends on its context length only; "Partition
 * ceiling": sparse plans keep a ceiling of 8) and Known Limitations item 2
 * (top-k, init-block and local-block settings).  The indexer that scores blocks
 * is not described; its scores are an input.
 *
 * For request r with S = context_lens[r] tokens and nb = ceil(S / block_size)
 * logical blocks (at most max_blocks_per_seq; a longer request raises
 * PA_DEVERR_BAD_PAGE in *device_errors and only its first max_blocks_per_seq
 * blocks exist): the first init_blocks and the last local_blocks blocks are
 * always selected; of the blocks between them, the top_k with the highest
 * block_scores[r * score_stride + b], scores ordered as their fp32 bit
 * patterns (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN) and equal scores
 * by the lower block index.  Row r of sel_block_tables [num_seqs][sel_stride]
 * receives block_tables[r][b] of the selected blocks b in ascending order, then
 * -1; sel_context_lens[r] the tokens they hold (the tail block counts
 * S - (nb - 1) * block_size).  A pa_decode with sel_block_tables
 * (max_blocks_per_seq = sel_stride) and sel_context_lens is then the sparse
 * decode: each request's token attends to the keys of its selected blocks.
 *
 * block_scores: device fp32, rows of score_stride >= max_blocks_per_seq
 * entries; may be NULL when top_k == 0.  Requires sel_stride >= init_blocks +
 * top_k + local_blocks, all counts >= 0, 1 <= num_seqs <= 4096.
 * device_errors: optional device uint32 (NULL: none).  One kernel on `stream`
 * on the current device; no allocation, no host synchronisation, so it may be
 * captured in a CUDA graph.  PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED on bad
 * arguments, PA_ERR_CUDA if the launch fails. */
int pa_sparse_select(const float* block_scores, int score_stride, const int32_t* context_lens,
                     const int32_t* block_tables, int max_blocks_per_seq, int num_seqs,
                     int block_size, int top_k, int init_blocks, int local_blocks,
                     int32_t* sel_block_tables, int sel_stride, int32_t* sel_context_lens,
                     uint32_t* device_errors, void* stream);

/* Size of the file-scope device array that pa_decode_static works in. */
#define PA_STATIC_SCRATCH_BYTES (32u << 20)

/* pa_decode_static: the work of pa_plan_refresh followed by pa_decode in one
 * call that allocates no device memory.  The source pages have no counterpart:
 * it exists for callers that cannot call cudaMalloc while decoding -- a serving
 * engine that hands nearly all HBM to its own KV-cache pool and caching
 * allocator at start-up, or a runtime that may not allocate device memory once
 * it serves -- and so cannot create a pa_plan.  It has no sliding window and no
 * sinks, and takes K in the PA_K_ROWS layout.
 *
 * Arguments mean what they mean for pa_plan_build and pa_decode; the plan
 * parameters (max_query_len, max_partitions, budget, kind) are passed per call
 * and the plan is rebuilt from context_lens / cu_query_lens every call, on
 * `stream`.  The plan arrays and fp32 partial results live in one static device
 * array of PA_STATIC_SCRATCH_BYTES (32 MiB) that every GPU loading this code
 * keeps until the process exits.  A batch whose plan and partial results need
 * more than that is rejected with PA_ERR_UNSUPPORTED; the need is the
 * pa_plan_build footprint, dominated by the fp32 partials:
 * Q x min(C x max_query_len, max_partitions x num_tokens) x Hq x (D + 1) x 4
 * bytes, with Q = 4 when the split kernel may cut slots into pieces (single
 * query row per request and C x Hkv <= 4 x SMs; dropped to 1 when that does
 * not fit) and 1 otherwise,
 * with capacity C = min(n x P, max(n, ceil(W / Hkv))), plus about C x 24 +
 * n x 16 bytes of plan (and a list of row chunks when max_query_len x Hq/Hkv
 * exceeds 32).
 * device_errors: optional device pointer to a uint32 that receives the
 * PA_DEVERR_* bits (the caller clears it); NULL uses a word inside the static
 * array, cleared at the start of every call and not readable by the caller.
 * The first call on a device looks up the array's device address there (with
 * that device current), so make it before any stream capture.  Every call
 * shares the array and it keeps the last call's contents: calls whose GPU work
 * can overlap (several streams or threads) race and must be serialised by the
 * caller.  Never calls cudaMalloc or cudaFree. */
int pa_decode_static(const void* q, int q_dtype, int num_tokens, int num_q_heads, int head_dim,
                     const void* k_cache, const void* v_cache, int kv_dtype, float k_scale,
                     float v_scale, int num_blocks, int num_kv_heads, int block_size,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, const int32_t* cu_query_lens, int num_seqs,
                     int max_query_len, int max_partitions, int budget, int kind, float scale,
                     void* out, uint32_t* device_errors, void* stream);

/* Host-side facts about a plan (any pointer may be NULL): its capacity C, the
 * batch size, the budget W and ceiling P actually used, the plan kind, the
 * device, and the bytes of device memory it owns. */
int pa_plan_info(const pa_plan* plan, int* capacity, int* num_seqs, int* budget,
                 int* max_partitions, int* kind, int* device, long long* device_bytes);

/* Copies the current work_info (capacity x 4 int32) and reduce_info
 * (num_seqs x 2 int32) to host memory, ordered after prior work on `stream`,
 * and waits for the copy (synchronises `stream`; not capturable); *capacity
 * receives C, the rows of work_info.  Any of the three destinations may be
 * NULL.  For tests and diagnostics. */
int pa_plan_download(const pa_plan* plan, int32_t* work_info, int32_t* reduce_info, int* capacity,
                     void* stream);

/* Reads the plan's sticky device error word (PA_DEVERR_* bits) into *errors,
 * ordered after prior work on `stream`; waits for it (synchronises `stream`;
 * not capturable).  clear != 0 resets the word to 0 afterwards. */
int pa_plan_read_errors(pa_plan* plan, uint32_t* errors, int clear, void* stream);

/* Profiling hook: when both are non-NULL, every later pa_decode records
 * start_event immediately before its split-KV kernel and stop_event right
 * after it, on the decode stream (cudaEvent_t values passed as void*; the
 * caller owns them).  NULL, NULL turns it off. */
int pa_plan_set_split_events(pa_plan* plan, void* start_event, void* stop_event);

/* Profiling hook: as pa_plan_set_split_events, but the events bracket the
 * whole pa_decode call (split-KV kernel and merge kernel).  Inside a stream
 * capture both hooks record external events, which fire on every replay. */
int pa_plan_set_call_events(pa_plan* plan, void* start_event, void* stop_event);

/* Releases the plan's device buffers and the plan (NULL is a no-op).  The
 * caller must ensure no enqueued work still uses the plan. */
int pa_plan_destroy(pa_plan* plan);

/* A static, human-readable name for a status code. */
const char* pa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
