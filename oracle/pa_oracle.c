/*
 * pa_oracle.c -- plain, slow fp64 CPU oracle for paged-KV GQA decode attention
 * and for the context-proportional work-plan rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or constant with the CUDA library: every number format
 * and formula below is written out here from its definition.
 *
 * Sources (web pages; cited by title and section):
 *   [ATOM-2366] ROCm/ATOM pull 2366, "[MiniMax-M3] Route the paged decode to
 *               aiter's FlyDSL kernel with work planner": sections 1
 *               (Motivation), 3 (Design), 5 (Test Result, "Planner drift at the
 *               real ceiling"), review item 3 (capacity formula), item 2
 *               (per-task begin/end tiles plus seq_ctx in the plan).
 *   [ATOM-2514] ROCm/ATOM pull 2514, "Fix(attention): adapt the FlyDSL paged
 *               decode to aiter #5809 (explicit work plans)": Motivation and
 *               Design ("aiter's default workgroup budget (2xCU)").
 *   [RDNA-29]   opengfx1030/vllm-rdna pull 29 (mixed and MTP-verify batches),
 *               Change section 1 "Kernel: per-token causal decode".
 *
 * Readings taken where the pages are silent (the same readings the CUDA path
 * implements, stated independently there):
 *   - partition tile T is a parameter (256 tokens in every caller);
 *   - proportional rule: reserve one partition per active request, share the
 *     remaining capacity in proportion to context length with floor rounding,
 *     clamp to min(max_partitions, ceil(S/T));
 *   - uniform comparator: every active request gets min(P, ceil(S/T),
 *     floor(C / n_active));
 *   - a request is active iff S > 0 and it owns at least one query row;
 *   - slots are request-major, partitions ascending, request r's ceil(S/T)
 *     tiles split as part j = [floor(j*nt/p), floor((j+1)*nt/p));
 *   - work_info words are (seq, tile_begin, tile_end, seq_ctx), seq = -1 for
 *     an unused slot; reduce_info words are (first_slot, num_parts), with
 *     first_slot the exclusive running sum of num_parts;
 *   - fp8 is OCP e4m3fn (bias 7, no infinities, S.1111.111 = NaN); a stored
 *     byte b means e4m3fn(b) * scale;
 *   - the kv head of q head hq is hq / (Hq / Hkv);
 *   - sliding window W > 0 ([RDNA-29] Change 1 applies the window to each
 *     token on its own): token i, which may see keys [0, K_i), sees only the W most
 *     recent of them, [max(0, K_i - W), K_i); W = 0 means no window;
 *   - with a window the plan sizes a request by the keys its tokens read: it
 *     starts at the tile holding the first token's first visible key and runs
 *     the rule on that range's length (tile indices stay absolute);
 *   - attention sinks (named in the pa_decode signature the pages quote): a
 *     logit per q head, in the units of scale * q.k, that joins the softmax
 *     denominator only: out = sum_j e^(s_j) v_j / (sum_j e^(s_j) + e^(sink));
 *   - K may also come in the 5-D layout [num_blocks, Hkv, D/16, block_size, 16]
 *     the pages' gate checks (the head dim in 16-element groups, each group's
 *     rows contiguous per page); V keeps [num_blocks, Hkv, block_size, D];
 *   - sparse top-k decode ([ATOM-2366] section 3, the sparse call sites read a
 *     fixed top-k window; [ATOM-2514] Design, "Once-per-step sparse refresh":
 *     the local tail block is always selected, so a row's length depends on
 *     seq_len only; Known Limitations item 2: top-k, init-block and
 *     local-block settings): the indexer that scores a request's blocks is not
 *     described, so its per-block fp32 scores are an input.  Of request r's
 *     nb = ceil(S / block_size) logical blocks, the first init_blocks and the
 *     last local_blocks are always selected, and of the others the top_k with
 *     the highest score, scores compared in the total order of their fp32 bit
 *     patterns (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN) and equal
 *     scores by the lower block index.  The selected blocks in ascending
 *     logical order make the request's sparse block-table row and its length
 *     is the tokens they hold (the tail block holds S - (nb - 1) * block_size).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 0, OR_FP16 = 1, OR_FP8_E4M3 = 2 };
enum { OR_PLAN_PROPORTIONAL = 0, OR_PLAN_UNIFORM = 1 };

/* ---------------------------------------------------------------- formats */

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double oracle_fp16_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: (m / 1024) * 2^-14 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp(1.0 + (double)m / 1024.0, e - 15);
  return s ? -v : v;
}

/* OCP float8 e4m3fn: 1 sign, 4 exponent (bias 7), 3 mantissa bits; the
 * all-ones exponent is an ordinary binade except mantissa 111 (NaN). */
double oracle_e4m3fn_to_double(uint8_t b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: (m / 8) * 2^-6 */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

static double load_q(const void* q, int dtype, int64_t idx) {
  const uint16_t* p = (const uint16_t*)q;
  return dtype == OR_FP16 ? oracle_fp16_to_double(p[idx]) : oracle_bf16_to_double(p[idx]);
}

static double load_kv(const void* cache, int dtype, int64_t idx, double scale) {
  if (dtype == OR_FP8_E4M3) return oracle_e4m3fn_to_double(((const uint8_t*)cache)[idx]) * scale;
  const uint16_t* p = (const uint16_t*)cache;
  return dtype == OR_FP16 ? oracle_fp16_to_double(p[idx]) : oracle_bf16_to_double(p[idx]);
}

/* ------------------------------------------------------------ work plan */

/* Capacity of a plan ([ATOM-2366] review item 3 and section 5):
 *   C = min(n * P, max(n, ceil(W / Hkv))).                              */
long long oracle_plan_capacity(int n, int num_kv_heads, int max_partitions, int budget) {
  long long per_head = ((long long)budget + num_kv_heads - 1) / num_kv_heads;
  long long floor_n = per_head > n ? per_head : n;
  long long cap = (long long)n * max_partitions;
  return cap < floor_n ? cap : floor_n;
}

/* Query rows of request r: L = cu[r+1] - cu[r], or 1 without cu ([RDNA-29]). */
static long long rows_of(const int32_t* cu, int r) {
  return cu ? (long long)cu[r + 1] - (long long)cu[r] : 1;
}

/* First tile a request's plan covers: 0 without a window; with one, the tile
 * holding the first visible key of its first query token. */
static long long first_tile(long long S, long long L, int window, int tile) {
  if (window <= 0) return 0;
  long long first_key = S - (L - 1) - window;
  if (first_key < 0) first_key = 0;
  return first_key / tile;
}

/* Builds the plan.  Returns the capacity C, or -1 if work_info has fewer than
 * C slots.  work_info is C x 4 int32, reduce_info is n x 2 int32.  With a
 * sliding window the rule runs on each request's planned range (see
 * first_tile); window = 0 is the plain rule. */
long long oracle_plan_window(int n, const int32_t* context_lens, const int32_t* cu,
                             int num_kv_heads, int max_partitions, int budget, int tile, int kind,
                             int window, int32_t* work_info, long long work_slots,
                             int32_t* reduce_info) {
  long long C = oracle_plan_capacity(n, num_kv_heads, max_partitions, budget);
  if (C > work_slots) return -1;

  /* the length the rule sees: from the first planned tile to S */
  long long n_act = 0, sum_s = 0;
  for (int r = 0; r < n; ++r) {
    long long S = context_lens[r], L = rows_of(cu, r);
    if (S > 0 && L > 0) {
      n_act += 1;
      sum_s += S - first_tile(S, L, window, tile) * tile;
    }
  }

  long long slot = 0;
  for (int r = 0; r < n; ++r) {
    long long S = context_lens[r], L = rows_of(cu, r);
    long long p = 0;
    if (S > 0 && L > 0) {
      long long t0 = first_tile(S, L, window, tile);
      long long len = S - t0 * tile;
      long long tiles = (len + tile - 1) / tile;
      long long share;
      if (kind == OR_PLAN_UNIFORM)
        share = C / n_act;                        /* same count for everyone */
      else
        share = 1 + ((C - n_act) * len) / sum_s;  /* proportional to the length */
      p = max_partitions;
      if (tiles < p) p = tiles;
      if (share < p) p = share;
      for (long long j = 0; j < p; ++j) {
        int32_t* w = work_info + 4 * (slot + j);
        w[0] = r;
        w[1] = (int32_t)(t0 + (j * tiles) / p);
        w[2] = (int32_t)(t0 + ((j + 1) * tiles) / p);
        w[3] = (int32_t)S;
      }
    }
    reduce_info[2 * r + 0] = (int32_t)slot;
    reduce_info[2 * r + 1] = (int32_t)p;
    slot += p;
  }
  for (; slot < C; ++slot) {
    int32_t* w = work_info + 4 * slot;
    w[0] = -1;
    w[1] = w[2] = w[3] = 0;
  }
  return C;
}

/* The pages' rule: no window. */
long long oracle_plan(int n, const int32_t* context_lens, const int32_t* cu, int num_kv_heads,
                      int max_partitions, int budget, int tile, int kind, int32_t* work_info,
                      long long work_slots, int32_t* reduce_info) {
  return oracle_plan_window(n, context_lens, cu, num_kv_heads, max_partitions, budget, tile,
                            kind, 0, work_info, work_slots, reduce_info);
}

/* ------------------------------------------------------------- attention */

/* Which request owns query row t; -1 for graph padding past cu[n]. */
static int owner_of(const int32_t* cu, int n, int t) {
  if (!cu) return t < n ? t : -1;
  for (int r = 0; r < n; ++r)
    if (cu[r] <= t && t < cu[r + 1]) return r;
  return -1;
}

struct kv_view {
  const void *k, *v;
  int dtype;
  double k_scale, v_scale;
  int num_kv_heads, block_size, head_dim, max_blocks;
  const int32_t* block_tables;
  int k_layout;  /* 0: [nb, Hkv, bs, D]; 1: [nb, Hkv, D/16, bs, 16] */
};

/* Flat element index of key j's row of request r, kv head h, in a cache laid
 * out [num_blocks, Hkv, block_size, D]. */
static int64_t key_row(const struct kv_view* kv, int r, int h, long long j) {
  int32_t page = kv->block_tables[(int64_t)r * kv->max_blocks + j / kv->block_size];
  return (((int64_t)page * kv->num_kv_heads + h) * kv->block_size + j % kv->block_size) *
         kv->head_dim;
}

/* Flat element index of element d of key j's K row of request r, kv head h. */
static int64_t key_elem(const struct kv_view* kv, int r, int h, long long j, int d) {
  if (kv->k_layout == 0) return key_row(kv, r, h, j) + d;
  int32_t page = kv->block_tables[(int64_t)r * kv->max_blocks + j / kv->block_size];
  int64_t slab = (int64_t)page * kv->num_kv_heads + h;  /* one (page, head): D/16 x bs x 16 */
  return ((slab * (kv->head_dim / 16) + d / 16) * kv->block_size + j % kv->block_size) * 16 +
         d % 16;
}

static double logit(const struct kv_view* kv, const void* q, int q_dtype, int64_t qoff, int r,
                    int h, long long j, double scale) {
  double dot = 0.0;
  for (int d = 0; d < kv->head_dim; ++d)
    dot += load_q(q, q_dtype, qoff + d) *
           load_kv(kv->k, kv->dtype, key_elem(kv, r, h, j, d), kv->k_scale);
  return scale * dot;
}

/* Key count of query row t ([RDNA-29] Change 1): token i of a request with L
 * query tokens and KV length S attends to keys [0, S - (L - 1 - i)). */
static long long keys_of_row(const int32_t* context_lens, const int32_t* cu, int r, int t) {
  long long L = rows_of(cu, r);
  long long i = cu ? t - cu[r] : 0;
  return (long long)context_lens[r] - (L - 1 - i);
}

/* First visible key of a row that sees keys below K: 0, or K - W with a window. */
static long long window_lo(long long K, int window) {
  if (window <= 0 || K <= window) return 0;
  return K - window;
}

/* Dense decode: the exact result, softmax(scale * q K^T) V per row and q head,
 * accumulated in fp64, over each row's visible keys [window_lo(K), K); a sink
 * (if given) adds e^(sink) to the denominator.  out is num_tokens x Hq x D
 * doubles.  Rows past cu[n], rows of a request with S <= 0 and rows with no
 * visible key are 0. */
void oracle_decode_ext(const void* q, int q_dtype, int num_tokens, int num_q_heads, int head_dim,
                       const void* k_cache, const void* v_cache, int kv_dtype, double k_scale,
                       double v_scale, int num_kv_heads, int block_size,
                       const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                       const int32_t* cu, int n, double scale, int window, const double* sinks,
                       int k_layout, double* out) {
  struct kv_view kv = {k_cache, v_cache, kv_dtype,
                       kv_dtype == OR_FP8_E4M3 ? k_scale : 1.0,
                       kv_dtype == OR_FP8_E4M3 ? v_scale : 1.0,
                       num_kv_heads, block_size, head_dim, max_blocks, block_tables, k_layout};
  int group = num_q_heads / num_kv_heads;
  long long total = (long long)num_tokens * num_q_heads;

#pragma omp parallel for schedule(dynamic, 1)
  for (long long th = 0; th < total; ++th) {
    int t = (int)(th / num_q_heads), hq = (int)(th % num_q_heads), h = hq / group;
    double* o = out + th * head_dim;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    int r = owner_of(cu, n, t);
    if (r < 0 || context_lens[r] <= 0) continue;
    long long K = keys_of_row(context_lens, cu, r, t);
    if (K <= 0) continue;
    long long lo = window_lo(K, window);

    double* s = (double*)malloc(sizeof(double) * (size_t)(K - lo));
    double m = -INFINITY, l = 0.0;
    for (long long j = lo; j < K; ++j) {
      s[j - lo] = logit(&kv, q, q_dtype, th * head_dim, r, h, j, scale);
      if (s[j - lo] > m) m = s[j - lo];
    }
    if (sinks && sinks[hq] > m) m = sinks[hq];
    for (long long j = lo; j < K; ++j) {
      double w = exp(s[j - lo] - m);
      int64_t vrow = key_row(&kv, r, h, j);
      l += w;
      for (int d = 0; d < head_dim; ++d)
        o[d] += w * load_kv(kv.v, kv.dtype, vrow + d, kv.v_scale);
    }
    if (sinks) l += exp(sinks[hq] - m);
    for (int d = 0; d < head_dim; ++d) o[d] /= l;
    free(s);
  }
}

/* No window, no sink. */
void oracle_decode(const void* q, int q_dtype, int num_tokens, int num_q_heads, int head_dim,
                   const void* k_cache, const void* v_cache, int kv_dtype, double k_scale,
                   double v_scale, int num_kv_heads, int block_size,
                   const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                   const int32_t* cu, int n, double scale, double* out) {
  oracle_decode_ext(q, q_dtype, num_tokens, num_q_heads, head_dim, k_cache, v_cache, kv_dtype,
                    k_scale, v_scale, num_kv_heads, block_size, block_tables, max_blocks,
                    context_lens, cu, n, scale, 0, NULL, 0, out);
}

/* Planned decode, computed the way the method computes it: each task of the
 * plan forms a partial softmax over its own tile range; a request's partials
 * are then combined with weights exp(lse_j - max lse) ([ATOM-2366] sections 3
 * and 6.5: split attention tile, then the "PS reduce").  Equal to
 * oracle_decode up to rounding for every valid plan. */
void oracle_decode_planned_ext(const void* q, int q_dtype, int num_tokens, int num_q_heads,
                               int head_dim, const void* k_cache, const void* v_cache,
                               int kv_dtype, double k_scale, double v_scale, int num_kv_heads,
                               int block_size, const int32_t* block_tables, int max_blocks,
                               const int32_t* context_lens, const int32_t* cu, int n,
                               double scale, const int32_t* work_info,
                               const int32_t* reduce_info, int tile, int window,
                               const double* sinks, int k_layout, double* out) {
  struct kv_view kv = {k_cache, v_cache, kv_dtype,
                       kv_dtype == OR_FP8_E4M3 ? k_scale : 1.0,
                       kv_dtype == OR_FP8_E4M3 ? v_scale : 1.0,
                       num_kv_heads, block_size, head_dim, max_blocks, block_tables, k_layout};
  int group = num_q_heads / num_kv_heads;
  long long total = (long long)num_tokens * num_q_heads;

#pragma omp parallel for schedule(dynamic, 1)
  for (long long th = 0; th < total; ++th) {
    int t = (int)(th / num_q_heads), hq = (int)(th % num_q_heads), h = hq / group;
    double* o = out + th * head_dim;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    int r = owner_of(cu, n, t);
    if (r < 0) continue;
    int first = reduce_info[2 * r], parts = reduce_info[2 * r + 1];
    if (parts <= 0) continue;
    long long K = keys_of_row(context_lens, cu, r, t);
    long long row_lo = window_lo(K, window);

    double* po = (double*)calloc((size_t)parts * head_dim, sizeof(double));
    double* lse = (double*)malloc(sizeof(double) * (size_t)parts);
    for (int j = 0; j < parts; ++j) {
      const int32_t* w = work_info + 4 * (first + j);
      long long lo = (long long)w[1] * tile, hi = (long long)w[2] * tile;
      if (hi > w[3]) hi = w[3];
      if (hi > K) hi = K;
      if (lo < row_lo) lo = row_lo;
      lse[j] = -INFINITY;
      if (lo >= hi) continue;
      double m = -INFINITY, l = 0.0;
      for (long long k = lo; k < hi; ++k) {
        double s = logit(&kv, q, q_dtype, th * head_dim, r, h, k, scale);
        if (s > m) m = s;
      }
      for (long long k = lo; k < hi; ++k) {
        double e = exp(logit(&kv, q, q_dtype, th * head_dim, r, h, k, scale) - m);
        int64_t vrow = key_row(&kv, r, h, k);
        l += e;
        for (int d = 0; d < head_dim; ++d)
          po[(size_t)j * head_dim + d] += e * load_kv(kv.v, kv.dtype, vrow + d, kv.v_scale);
      }
      for (int d = 0; d < head_dim; ++d) po[(size_t)j * head_dim + d] /= l;
      lse[j] = m + log(l);
    }
    double M = -INFINITY;
    for (int j = 0; j < parts; ++j)
      if (lse[j] > M) M = lse[j];
    if (M > -INFINITY) {
      if (sinks && sinks[hq] > M) M = sinks[hq];
      double wsum = 0.0;
      for (int j = 0; j < parts; ++j) {
        if (lse[j] == -INFINITY) continue;
        double w = exp(lse[j] - M);
        wsum += w;
        for (int d = 0; d < head_dim; ++d) o[d] += w * po[(size_t)j * head_dim + d];
      }
      if (sinks) wsum += exp(sinks[hq] - M);  /* the sink joins the merge once */
      for (int d = 0; d < head_dim; ++d) o[d] /= wsum;
    }
    free(po);
    free(lse);
  }
}

/* No window, no sink. */
void oracle_decode_planned(const void* q, int q_dtype, int num_tokens, int num_q_heads,
                           int head_dim, const void* k_cache, const void* v_cache, int kv_dtype,
                           double k_scale, double v_scale, int num_kv_heads, int block_size,
                           const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, const int32_t* cu, int n, double scale,
                           const int32_t* work_info, const int32_t* reduce_info, int tile,
                           double* out) {
  oracle_decode_planned_ext(q, q_dtype, num_tokens, num_q_heads, head_dim, k_cache, v_cache,
                            kv_dtype, k_scale, v_scale, num_kv_heads, block_size, block_tables,
                            max_blocks, context_lens, cu, n, scale, work_info, reduce_info, tile,
                            0, NULL, 0, out);
}

/* ------------------------------------------------------ sparse top-k select */

/* The fp32 total order as an unsigned key: flip every bit of a negative
 * pattern, set the sign bit of a non-negative one. */
static uint32_t order_key(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

typedef struct {
  uint32_t key;
  int block;
} scored_block;

/* Higher key first, then lower block index. */
static int by_score_then_index(const void* a, const void* b) {
  const scored_block* x = (const scored_block*)a;
  const scored_block* y = (const scored_block*)b;
  if (x->key != y->key) return x->key > y->key ? -1 : 1;
  return (x->block > y->block) - (x->block < y->block);
}

/* Selection for every request (see the reading above).  scores: row r holds
 * the scores of r's logical blocks at [r * score_stride, ...); may be NULL when
 * top_k == 0.  Blocks at or past max_blocks do not exist for the selection.
 * sel_tables [num_seqs][sel_stride] receives the physical blocks (block_tables
 * entries) of the selected logical blocks in ascending order, -1 after them;
 * sel_lens[r] the tokens they hold.  Returns the largest selection size. */
int oracle_sparse_select(const float* scores, int score_stride, const int32_t* context_lens,
                         const int32_t* block_tables, int max_blocks, int num_seqs,
                         int block_size, int top_k, int init_blocks, int local_blocks,
                         int32_t* sel_tables, int sel_stride, int32_t* sel_lens) {
  int most = 0;
  unsigned char* take = (unsigned char*)malloc(max_blocks > 0 ? (size_t)max_blocks : 1);
  scored_block* cand = (scored_block*)malloc(sizeof(scored_block) * (max_blocks > 0 ? max_blocks : 1));
  for (int r = 0; r < num_seqs; ++r) {
    const long long S = context_lens[r] > 0 ? context_lens[r] : 0;
    long long nb_all = (S + block_size - 1) / block_size;
    const int nb = (int)(nb_all < max_blocks ? nb_all : max_blocks);
    int ncand = 0;
    for (int b = 0; b < nb; ++b) {
      const int fixed = b < init_blocks || b >= nb - local_blocks;
      take[b] = (unsigned char)fixed;
      if (!fixed) {  /* scores are read only when some are chosen by them */
        cand[ncand].key = top_k > 0 ? order_key(scores[(size_t)r * score_stride + b]) : 0u;
        cand[ncand].block = b;
        ++ncand;
      }
    }
    qsort(cand, (size_t)ncand, sizeof(scored_block), by_score_then_index);
    for (int i = 0; i < ncand && i < top_k; ++i) take[cand[i].block] = 1;
    int count = 0;
    long long tokens = 0;
    for (int b = 0; b < nb; ++b) {
      if (!take[b]) continue;
      if (count < sel_stride)
        sel_tables[(size_t)r * sel_stride + count] = block_tables[(size_t)r * max_blocks + b];
      ++count;
      const long long end = (long long)(b + 1) * block_size < S ? (long long)(b + 1) * block_size : S;
      tokens += end - (long long)b * block_size;
    }
    for (int i = count; i < sel_stride; ++i) sel_tables[(size_t)r * sel_stride + i] = -1;
    sel_lens[r] = (int32_t)tokens;
    if (count > most) most = count;
  }
  free(take);
  free(cand);
  return most;
}

/* Threads an OpenMP region of this library uses (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
