// pa_sparse.cu -- sparse top-k block selection: for every request, the block
// table of the KV blocks a sparse decode reads and the number of tokens they
// hold.
//
// "[MiniMax-M3] Route the paged decode to aiter's FlyDSL kernel with work
// planner", section 3: the sparse call sites read a fixed top-k window.
// "Fix(attention): adapt the FlyDSL paged decode to aiter #5809 (explicit work
// plans)", Design ("Once-per-step sparse refresh", "Partition ceiling") and
// Known Limitations item 2: the local tail block is always selected, so a
// request's selected length depends only on its context length; the settings
// are top-k, init blocks and local blocks; sparse plans keep a ceiling of 8.
// The indexer that scores blocks is not described: its per-block fp32 scores
// are an input.  Of request r's nb = ceil(S / bs) logical blocks the first
// init_blocks and the last local_blocks are always taken; of the blocks
// between them, the top_k with the highest score -- scores ordered as their
// fp32 bit patterns (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN), equal
// scores by the lower block index.  The taken blocks in ascending logical
// order form the request's sparse block-table row (their physical blocks,
// then -1), and its length is the tokens they hold.
//
// One CTA per request.  The candidates' 32-bit order keys are read once into
// shared memory (up to kSelSmemKeys of them; longer rows re-read global
// memory).  The top_k-th largest key T is found by a radix select over them
// (four 8-bit digits, shared-memory histograms).  A final pass in block order
// takes every fixed block, every candidate above T and the first `need`
// candidates equal to T; a block's place in the row is (fixed and larger
// blocks before it) + min(equal blocks before it, need), counted with warp
// ballots over each warp's run of blocks and one barrier for the warp totals,
// so the row comes out sorted.  No sort, no global scratch, no host
// synchronisation.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelSmemKeys = 8192;  // candidate keys cached in shared memory (32 KB)

struct SelectParams {
  const float* scores;
  long long score_stride;
  const int32_t* context_lens;
  const int32_t* block_tables;
  int max_blocks;
  int bs;
  int top_k;
  int init_blocks;
  int local_blocks;
  int32_t* sel_tables;
  int sel_stride;
  int32_t* sel_lens;
  unsigned* err;
};

// fp32 total order as an unsigned key, from the score's bit pattern (loaded
// as an integer: no floating-point operation touches it, so NaN payloads and
// signs are kept).
__device__ __forceinline__ uint32_t order_key(uint32_t u) {
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kSelThreads) sparse_select_kernel(const SelectParams p) {
  __shared__ int s_hist[2][256];  // digit histograms, alternating by pass
  __shared__ int s_wbig[kSelWarps], s_weq[kSelWarps];
  __shared__ uint32_t s_prefix[2];  // alternating by pass
  __shared__ int s_remaining[2];
  __shared__ int s_tail;
  extern __shared__ uint32_t s_keys[];  // min(max_blocks, kSelSmemKeys) entries
  pdl_trigger();  // the planner may be scheduled; it waits for these lengths
  pdl_wait();     // the scores (an indexer's output) are complete

  const int r = blockIdx.x;
  const long long S = p.context_lens[r] > 0 ? p.context_lens[r] : 0;
  const long long nb_all = (S + p.bs - 1) / p.bs;
  const int nb = static_cast<int>(nb_all < p.max_blocks ? nb_all : p.max_blocks);
  if (nb_all > p.max_blocks && threadIdx.x == 0 && p.err) atomicOr(p.err, PA_DEVERR_BAD_PAGE);
  // candidates: the blocks between the init and the local ones, [lo, hi)
  const int lo = min(p.init_blocks, nb);
  const int hi = max(lo, nb - p.local_blocks);
  const int ncand = hi - lo;
  const int k = min(p.top_k, ncand);
  const bool partial = k > 0 && k < ncand;  // else all candidates or none are taken
  const uint32_t* sc = reinterpret_cast<const uint32_t*>(p.scores) +
                       static_cast<long long>(r) * p.score_stride;
  const bool cached = ncand <= kSelSmemKeys;
  auto key_at = [&](int b) { return cached ? s_keys[b - lo] : order_key(__ldg(sc + b)); };
  if (partial && cached)
    for (int b = lo + threadIdx.x; b < hi; b += kSelThreads) s_keys[b - lo] = order_key(__ldg(sc + b));
  for (int i = threadIdx.x; i < 256; i += kSelThreads) s_hist[0][i] = 0;
  __syncthreads();  // the keys and the first histogram are ready

  // ---- radix select: T = the k-th largest candidate key, need = how many
  // candidates equal to T are taken (the k - need larger ones all are)
  uint32_t T = 0u;
  int need = 0;
  if (partial) {
    uint32_t prefix = 0u, mask = 0u;
    int remaining = k;
    for (int pass = 0, shift = 24; shift >= 0; ++pass, shift -= 8) {
      // Histogram pass `pass` fills s_hist[pass & 1] (zeroed one pass ahead)
      // and zeroes the other one, whose last readers finished a barrier ago.
      int* hist = s_hist[pass & 1];
      for (int i = threadIdx.x; i < 256; i += kSelThreads) s_hist[(pass + 1) & 1][i] = 0;
      for (int b = lo + threadIdx.x; b < hi; b += kSelThreads) {
        const uint32_t key = key_at(b);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l holds digits 255 - 8l down to 248 - 8l; find the digit where
        // the count from the top reaches `remaining`
        const int lane = threadIdx.x;
        int c[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[255 - 8 * lane - j];
          sum += c[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int excl = incl - sum;
        const bool mine = excl < remaining && remaining <= incl;
        const unsigned who = __ballot_sync(0xffffffffu, mine);
        if (mine && lane == __ffs(who) - 1) {
          int acc = excl, d = 255 - 8 * lane;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (acc + c[j] >= remaining) {
              d = 255 - 8 * lane - j;
              break;
            }
            acc += c[j];
          }
          s_prefix[pass & 1] = prefix | (static_cast<uint32_t>(d) << shift);
          s_remaining[pass & 1] = remaining - acc;
        }
      }
      __syncthreads();  // (the next pass writes the other s_prefix / s_remaining)
      prefix = s_prefix[pass & 1];
      remaining = s_remaining[pass & 1];
      mask |= 0xFFu << shift;
    }
    T = prefix;
    need = remaining;
  }

  // ---- take and compact, in block order.  Per block: big = fixed, or a
  // candidate taken whole or above T; eq = a candidate equal to T.  A block is
  // taken if big, or eq and fewer than `need` eq blocks precede it; its place
  // in the row is (big blocks before it) + min(eq blocks before it, need).
  // Warp w owns a contiguous run of 32-block chunks: a first pass counts its
  // big and eq blocks (ballots), one barrier publishes the warp totals, and a
  // second pass places the blocks from the totals of the warps before it.
  int32_t* row = p.sel_tables + static_cast<long long>(r) * p.sel_stride;
  const int32_t* bt = p.block_tables + static_cast<long long>(r) * p.max_blocks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;  // lanes below this one
  const int chunks = (nb + 31) / 32;
  const int cpw = (chunks + kSelWarps - 1) / kSelWarps;  // chunks per warp
  const int c_lo = min(chunks, warp * cpw), c_hi = min(chunks, c_lo + cpw);
  auto flags = [&](int b, bool& big, bool& eq) {
    const bool in = b < nb;
    const bool cand = in && b >= lo && b < hi;
    big = in && (!cand || k == ncand);
    eq = false;
    if (partial && cand) {
      const uint32_t key = key_at(b);
      big = key > T;
      eq = key == T;
    }
  };
  int my_big = 0, my_eq = 0;
  for (int c = c_lo; c < c_hi; ++c) {
    bool big, eq;
    flags(c * 32 + lane, big, eq);
    my_big += __popc(__ballot_sync(0xffffffffu, big));
    my_eq += __popc(__ballot_sync(0xffffffffu, eq));
  }
  if (lane == 0) {
    s_wbig[warp] = my_big;
    s_weq[warp] = my_eq;
  }
  if (threadIdx.x == 0) s_tail = 0;
  __syncthreads();
  int big_base = 0, eq_base = 0, big_all = 0, eq_all = 0;
#pragma unroll
  for (int v = 0; v < kSelWarps; ++v) {
    const int wb = s_wbig[v], we = s_weq[v];
    if (v < warp) {
      big_base += wb;
      eq_base += we;
    }
    big_all += wb;
    eq_all += we;
  }
  for (int c = c_lo; c < c_hi; ++c) {
    const int b = c * 32 + lane;
    bool big, eq;
    flags(b, big, eq);
    const unsigned bb = __ballot_sync(0xffffffffu, big), be = __ballot_sync(0xffffffffu, eq);
    const int eq_before = eq_base + __popc(be & lt);
    if (big || (eq && eq_before < need)) {
      row[big_base + __popc(bb & lt) + min(eq_before, need)] = __ldg(bt + b);
      if (b == nb_all - 1) s_tail = 1;  // the request's last, possibly partial, block
    }
    big_base += __popc(bb);
    eq_base += __popc(be);
  }
  const int taken = big_all + min(eq_all, need);
  for (int i = taken + threadIdx.x; i < p.sel_stride; i += kSelThreads) row[i] = -1;
  __syncthreads();
  if (threadIdx.x == 0) {
    const long long short_by = s_tail ? nb_all * p.bs - S : 0;  // empty slots of the tail block
    p.sel_lens[r] = static_cast<int32_t>(static_cast<long long>(taken) * p.bs - short_by);
  }
}

}  // namespace

}  // namespace pa

extern "C" int pa_sparse_select(const float* block_scores, int score_stride,
                                const int32_t* context_lens, const int32_t* block_tables,
                                int max_blocks_per_seq, int num_seqs, int block_size, int top_k,
                                int init_blocks, int local_blocks, int32_t* sel_block_tables,
                                int sel_stride, int32_t* sel_context_lens,
                                uint32_t* device_errors, void* stream) {
  if (!context_lens || !block_tables || !sel_block_tables || !sel_context_lens)
    return PA_ERR_INVALID_ARG;
  if (num_seqs < 1 || max_blocks_per_seq < 1 || block_size < 1 || top_k < 0 ||
      init_blocks < 0 || local_blocks < 0 || sel_stride < 1)
    return PA_ERR_INVALID_ARG;
  if (top_k > 0 && (!block_scores || score_stride < max_blocks_per_seq)) return PA_ERR_INVALID_ARG;
  if (static_cast<long long>(init_blocks) + top_k + local_blocks > sel_stride)
    return PA_ERR_INVALID_ARG;
  if (num_seqs > PA_MAX_SEQS) return PA_ERR_UNSUPPORTED;
  pa::SelectParams sp;
  sp.scores = block_scores;
  sp.score_stride = top_k > 0 ? score_stride : 0;
  sp.context_lens = context_lens;
  sp.block_tables = block_tables;
  sp.max_blocks = max_blocks_per_seq;
  sp.bs = block_size;
  sp.top_k = top_k;
  sp.init_blocks = init_blocks;
  sp.local_blocks = local_blocks;
  sp.sel_tables = sel_block_tables;
  sp.sel_stride = sel_stride;
  sp.sel_lens = sel_context_lens;
  sp.err = device_errors;
  const int cache = max_blocks_per_seq < pa::kSelSmemKeys ? max_blocks_per_seq : pa::kSelSmemKeys;
  const cudaError_t e = pa::launch_pdl(pa::sparse_select_kernel, dim3(num_seqs),
                                       dim3(pa::kSelThreads), cache * 4,
                                       static_cast<cudaStream_t>(stream), sp);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
