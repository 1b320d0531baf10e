// moe_align_block_size: stable counting sort of the (token, expert) pairs by
// expert, each expert's segment padded to a multiple of block_m.
//
// Follows the mini-sglang MoE chapter ("fused MoE", moe_align_block_size):
// counts per expert, padded lengths, exclusive prefix sum, stable placement of
// every pair at seg_start[e] + rank-within-expert, sentinel num_pairs in the
// padding, the expert of every block.
//
// Two kernels over chunks of S consecutive pairs (one CTA per chunk):
//  1. count: per-chunk expert histogram (shared-memory atomics; counts do not
//     depend on order) written to the workspace; the last CTA to finish (a
//     ticket taken after a fence) scans the histograms: per-expert totals,
//     padded lengths, segment starts, and for every chunk the position where its
//     first pair of each expert lands. It also writes offsets, the padded
//     length, the block experts and the sentinels.
//  2. scatter: each chunk is re-read in order. Warp w owns a contiguous slice;
//     a shared [warp][expert] table gives each warp's write cursors; walking its
//     slice 32 pairs at a time, __match_any_sync groups lanes with the same
//     expert and a pair's rank among them is the popcount of its lower peers.
// Walking every range in order makes the sort stable; no atomics decide
// positions. Optionally (the fused forward) the token of every sorted position,
// pair / topk or -1 for padding, is written alongside, so that the grouped GEMMs
// read gather rows without a division. The first kernel also zeroes one word
// for the caller (the fused forward's gate_up tile counter), so that the
// following kernel on the stream starts from zero without a separate launch.
#include "common.cuh"

#include <algorithm>

namespace moe {
namespace {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kMaxChunks = 512;

struct AlignPlan {
  int chunk;    // pairs per chunk (multiple of 1024)
  int nchunks;
};

AlignPlan align_plan(int num_pairs) {
  AlignPlan p;
  const int per = std::max(1, (num_pairs + kMaxChunks * 1024 - 1) / (kMaxChunks * 1024));
  p.chunk = 1024 * per;
  p.nchunks = std::max(1, (num_pairs + p.chunk - 1) / p.chunk);
  return p;
}

__global__ void __launch_bounds__(kAlignThreads)
    align_count_scan_kernel(const int32_t* __restrict__ ids, int num_pairs, int E, int block_m, int cap, int chunk,
                            int nchunks, int32_t* __restrict__ chunk_base, int* __restrict__ done,
                            int32_t* __restrict__ sorted_ids, int32_t* __restrict__ sorted_tok,
                            int32_t* __restrict__ expert_ids, int32_t* __restrict__ expert_offsets,
                            int32_t* __restrict__ ntpp, int* __restrict__ err, int* __restrict__ zero_word) {
  pdl_trigger();
  pdl_wait();
  __shared__ int hist[MOE_MAX_EXPERTS];
  __shared__ int warp_tot[kAlignWarps];
  __shared__ int is_last;
  // the last CTA reuses hist for the segment starts, and keeps counts and padded lengths
  __shared__ int seg_count[MOE_MAX_EXPERTS];
  __shared__ int seg_padded[MOE_MAX_EXPERTS];
  int* seg_start = hist;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (zero_word && blockIdx.x == 0 && tid == 0) *zero_word = 0;
  for (int e = tid; e < E; e += kAlignThreads) hist[e] = 0;
  __syncthreads();
  const int lo = blockIdx.x * chunk;
  const int hi = min(num_pairs, lo + chunk);
  for (int p = lo + tid; p < hi; p += kAlignThreads) {
    const int e = __ldg(ids + p);
    if (e < 0 || e >= E) report_error(err, MOE_DEVERR_EXPERT_ID);
    else atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kAlignThreads) chunk_base[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(done, 1) == nchunks - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // Last CTA: totals, padded segments, per-chunk bases. One expert per thread
  // (E <= 1024) for the scans; the chunk histograms are read kBatch at a time
  // before any of them is overwritten (a load of one slot after the store to the
  // previous one would wait a full L2 round trip per chunk).
  constexpr int kBatch = 16;
  int count = 0, padded = 0;
  if (tid < E) {
    int c = 0;
    for (; c + kBatch <= nchunks; c += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) v[j] = __ldcg(chunk_base + static_cast<size_t>(c + j) * E + tid);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) count += v[j];
    }
    for (; c < nchunks; ++c) count += __ldcg(chunk_base + static_cast<size_t>(c) * E + tid);
    padded = (count + block_m - 1) / block_m * block_m;
  }
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int start = incl - padded + (warp > 0 ? warp_tot[warp - 1] : 0);
  const int total = warp_tot[kAlignWarps - 1];
  if (tid < E) {
    expert_offsets[tid] = start;
    seg_start[tid] = start;
    seg_count[tid] = count;
    seg_padded[tid] = padded;
    int run = start;
    int c = 0;
    for (; c + kBatch <= nchunks; c += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) v[j] = __ldcg(chunk_base + static_cast<size_t>(c + j) * E + tid);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        chunk_base[static_cast<size_t>(c + j) * E + tid] = run;
        run += v[j];
      }
    }
    for (; c < nchunks; ++c) {
      int32_t* slot = chunk_base + static_cast<size_t>(c) * E + tid;
      const int n = __ldcg(slot);
      *slot = run;
      run += n;
    }
  }
  if (tid == 0) {
    expert_offsets[E] = total;
    *ntpp = total;
  }
  __syncthreads();
  // block experts and padding sentinels: one warp per expert
  for (int e = warp; e < E; e += kAlignWarps) {
    const int st = seg_start[e], cnt = seg_count[e], pd = seg_padded[e];
    for (int blk = st / block_m + lane; blk < (st + pd) / block_m; blk += 32) expert_ids[blk] = e;
    for (int pos = st + cnt + lane; pos < st + pd; pos += 32) {
      sorted_ids[pos] = num_pairs;
      if (sorted_tok) sorted_tok[pos] = -1;
    }
  }
  for (int pos = total + tid; pos < cap; pos += kAlignThreads) {
    sorted_ids[pos] = num_pairs;
    if (sorted_tok) sorted_tok[pos] = -1;
  }
  for (int blk = total / block_m + tid; blk < cap / block_m; blk += kAlignThreads) expert_ids[blk] = -1;
}

__global__ void __launch_bounds__(kAlignThreads)
    align_scatter_kernel(const int32_t* __restrict__ ids, int num_pairs, int E, int chunk,
                         const int32_t* __restrict__ chunk_base, int* __restrict__ done,
                         int32_t* __restrict__ sorted_ids, int32_t* __restrict__ sorted_tok, int topk) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int cur[];  // [kAlignWarps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) cur[i] = 0;
  if (blockIdx.x == 0 && tid == 0) *done = 0;  // the count kernel of the next call starts from zero
  __syncthreads();
  const int lo = blockIdx.x * chunk;
  const int span = chunk / kAlignWarps;  // multiple of 32
  const int wlo = min(num_pairs, lo + warp * span);
  const int whi = min(num_pairs, wlo + span);
  // per-warp counts of its slice
  for (int b = wlo; b < whi; b += 32) {
    const int p = b + lane;
    const int v = (p < whi) ? __ldg(ids + p) : -1;
    if (v >= 0 && v < E) atomicAdd(&cur[warp * E + v], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = __ldg(chunk_base + static_cast<size_t>(blockIdx.x) * E + e);
    for (int w = 0; w < kAlignWarps; ++w) {
      const int n = cur[w * E + e];
      cur[w * E + e] = run;
      run += n;
    }
  }
  __syncthreads();
  for (int b = wlo; b < whi; b += 32) {
    const int p = b + lane;
    int e = (p < whi) ? __ldg(ids + p) : -1;
    if (e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int base = 0;
    if (e >= 0) base = cur[warp * E + e];
    __syncwarp();
    if (e >= 0) {
      sorted_ids[base + __popc(peers & lt_mask)] = p;
      if (sorted_tok) sorted_tok[base + __popc(peers & lt_mask)] = p / topk;
      if ((peers & lt_mask) == 0) cur[warp * E + e] = base + __popc(peers);
    }
    __syncwarp();
  }
}

// Small problems (chunk histograms x experts <= kSmallScan): the count kernel
// only writes each chunk's histogram, and every CTA of the scatter kernel reads
// all of them (at most 256 KB from L2) and derives in shared memory the expert
// totals, the padded segment starts and its own chunk's bases, so that no CTA
// waits for a last one to finish the scan.
constexpr int kSmallScan = 65536;

__global__ void __launch_bounds__(kAlignThreads)
    align_hist_kernel(const int32_t* __restrict__ ids, int num_pairs, int E, int chunk,
                      int32_t* __restrict__ hists, int* __restrict__ err, int* __restrict__ zero_word) {
  pdl_trigger();
  pdl_wait();
  __shared__ int hist[MOE_MAX_EXPERTS];
  const int tid = threadIdx.x;
  if (zero_word && blockIdx.x == 0 && tid == 0) *zero_word = 0;
  for (int e = tid; e < E; e += kAlignThreads) hist[e] = 0;
  __syncthreads();
  const int lo = blockIdx.x * chunk;
  const int hi = min(num_pairs, lo + chunk);
  for (int p = lo + tid; p < hi; p += kAlignThreads) {
    const int e = __ldg(ids + p);
    if (e < 0 || e >= E) report_error(err, MOE_DEVERR_EXPERT_ID);
    else atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kAlignThreads) hists[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];
}

// The histogram rows may be finer than the chunks (rows_per_chunk rows of chunk /
// rows_per_chunk pairs each, e.g. the per-tile counts written by the routing kernel).
__global__ void __launch_bounds__(kAlignThreads)
    align_scan_scatter_kernel(const int32_t* __restrict__ ids, int num_pairs, int E, int block_m, int cap, int chunk,
                              int nchunks, const int32_t* __restrict__ hists, int nrows, int rows_per_chunk,
                              int32_t* __restrict__ sorted_ids, int32_t* __restrict__ sorted_tok, int topk,
                              int32_t* __restrict__ expert_ids, int32_t* __restrict__ expert_offsets,
                              int32_t* __restrict__ ntpp, int* __restrict__ zero_word) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sm[];
  int* cur = sm;                              // [kAlignWarps][E] write cursors
  int* tot = cur + kAlignWarps * E;           // [E] pairs per expert
  int* bef = tot + E;                         // [E] pairs of the expert in earlier chunks
  int* seg = bef + E;                         // [E] padded segment starts
  __shared__ int warp_tot[kAlignWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (zero_word && blockIdx.x == 0 && tid == 0) *zero_word = 0;
  for (int i = tid; i < (kAlignWarps + 2) * E; i += kAlignThreads) sm[i] = 0;
  __syncthreads();
  // per-expert totals and counts in earlier chunks: thread (part, e) sums rows part, part + parts, ...
  // in registers, then the parts meet in shared memory (parts atomics per expert)
  {
    const int parts = kAlignThreads / E > 0 ? kAlignThreads / E : 1;
    const int part = tid / E, e = tid - part * E;
    if (part < parts) {
      const int split = static_cast<int>(blockIdx.x) * rows_per_chunk;  // rows before this chunk
      int t_sum = 0, b_sum = 0;
#pragma unroll 4
      for (int row = part; row < nrows; row += parts) {
        const int v = __ldcg(hists + static_cast<size_t>(row) * E + e);
        t_sum += v;
        b_sum += row < split ? v : 0;
      }
      if (t_sum) atomicAdd(&tot[e], t_sum);
      if (b_sum) atomicAdd(&bef[e], b_sum);
    }
  }
  __syncthreads();
  // padded lengths -> exclusive scan over experts (one expert per thread, E <= 1024)
  const int count = tid < E ? tot[tid] : 0;
  const int padded = (count + block_m - 1) / block_m * block_m;
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int start = incl - padded + (warp > 0 ? warp_tot[warp - 1] : 0);
  const int total = warp_tot[kAlignWarps - 1];
  if (tid < E) seg[tid] = start;
  if (blockIdx.x == 0) {
    if (tid < E) expert_offsets[tid] = start;
    if (tid == 0) {
      expert_offsets[E] = total;
      *ntpp = total;
    }
  }
  __syncthreads();
  // block experts and padding sentinels, spread over the grid (one SM alone is
  // store-bound on them): one warp per expert, experts and tail strided by CTA
  for (int e = static_cast<int>(blockIdx.x) * kAlignWarps + warp; e < E; e += nchunks * kAlignWarps) {
    const int st = seg[e], cnt = tot[e];
    const int pd = (cnt + block_m - 1) / block_m * block_m;
    for (int blk = st / block_m + lane; blk < (st + pd) / block_m; blk += 32) expert_ids[blk] = e;
    for (int pos = st + cnt + lane; pos < st + pd; pos += 32) {
      sorted_ids[pos] = num_pairs;
      if (sorted_tok) sorted_tok[pos] = -1;
    }
  }
  const int g0 = static_cast<int>(blockIdx.x) * kAlignThreads + tid, gstride = nchunks * kAlignThreads;
  for (int pos = total + g0; pos < cap; pos += gstride) {
    sorted_ids[pos] = num_pairs;
    if (sorted_tok) sorted_tok[pos] = -1;
  }
  for (int blk = total / block_m + g0; blk < cap / block_m; blk += gstride) expert_ids[blk] = -1;
  // stable scatter of this chunk (as in align_scatter_kernel)
  const int lo = blockIdx.x * chunk;
  const int span = chunk / kAlignWarps;  // multiple of 32
  const int wlo = min(num_pairs, lo + warp * span);
  const int whi = min(num_pairs, wlo + span);
  for (int b = wlo; b < whi; b += 32) {
    const int p = b + lane;
    const int v = (p < whi) ? __ldg(ids + p) : -1;
    if (v >= 0 && v < E) atomicAdd(&cur[warp * E + v], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = seg[e] + bef[e];
    for (int w = 0; w < kAlignWarps; ++w) {
      const int n = cur[w * E + e];
      cur[w * E + e] = run;
      run += n;
    }
  }
  __syncthreads();
  for (int b = wlo; b < whi; b += 32) {
    const int p = b + lane;
    int e = (p < whi) ? __ldg(ids + p) : -1;
    if (e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int base = 0;
    if (e >= 0) base = cur[warp * E + e];
    __syncwarp();
    if (e >= 0) {
      sorted_ids[base + __popc(peers & lt_mask)] = p;
      if (sorted_tok) sorted_tok[base + __popc(peers & lt_mask)] = p / topk;
      if ((peers & lt_mask) == 0) cur[warp * E + e] = base + __popc(peers);
    }
    __syncwarp();
  }
}

}  // namespace

size_t align_max_padded(int num_pairs, int E, int block_m) {
  if (num_pairs < 0 || E < 1 || block_m < 1) return 0;
  const size_t cap = static_cast<size_t>(num_pairs) + static_cast<size_t>(std::min(E, num_pairs)) * (block_m - 1);
  return align_up(cap, static_cast<size_t>(block_m));
}

bool valid_block_m(int bm) { return bm >= 1 && bm <= 256 && (bm & (bm - 1)) == 0; }

// Scratch of the align kernels: the completion ticket (256 bytes), then the chunk histograms.
size_t align_scratch_bytes(int num_pairs, int E) {
  const AlignPlan p = align_plan(num_pairs);
  return 256 + align_up(static_cast<size_t>(p.nchunks) * E * 4, 256);
}

moe_status_t launch_align(const int32_t* ids, int num_pairs, int E, int block_m, int32_t* sorted_ids,
                          int32_t* expert_ids, int32_t* expert_offsets, int32_t* ntpp, void* scratch, int* err,
                          cudaStream_t s, int32_t* sorted_tok, int topk, int* zero_word) {
  const int cap = static_cast<int>(align_max_padded(num_pairs, E, block_m));
  const AlignPlan p = align_plan(num_pairs);
  int* done = static_cast<int*>(scratch);
  int32_t* chunk_base = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(scratch) + 256);
  if (p.nchunks * E <= kSmallScan) {
    moe_status_t st = launch_pdl(align_hist_kernel, dim3(p.nchunks), dim3(kAlignThreads), 0, s, ids, num_pairs, E,
                                 p.chunk, chunk_base, err, zero_word);
    if (st != MOE_OK) return st;
    const size_t smem = static_cast<size_t>(kAlignWarps + 3) * E * sizeof(int);
    if (!ensure_smem_attr(reinterpret_cast<const void*>(align_scan_scatter_kernel),
                          static_cast<int>(static_cast<size_t>(kAlignWarps + 3) * MOE_MAX_EXPERTS * sizeof(int))))
      return MOE_ERR_CUDA;
    return launch_pdl(align_scan_scatter_kernel, dim3(p.nchunks), dim3(kAlignThreads), smem, s, ids, num_pairs, E,
                      block_m, cap, p.chunk, p.nchunks, static_cast<const int32_t*>(chunk_base), p.nchunks, 1,
                      sorted_ids, sorted_tok, topk > 0 ? topk : 1, expert_ids, expert_offsets, ntpp,
                      static_cast<int*>(nullptr));
  }
  moe_status_t st = launch_pdl(align_count_scan_kernel, dim3(p.nchunks), dim3(kAlignThreads), 0, s, ids, num_pairs,
                               E, block_m, cap, p.chunk, p.nchunks, chunk_base, done, sorted_ids, sorted_tok,
                               expert_ids, expert_offsets, ntpp, err, zero_word);
  if (st != MOE_OK) return st;
  const size_t smem = static_cast<size_t>(kAlignWarps) * E * sizeof(int);
  if (!ensure_smem_attr(reinterpret_cast<const void*>(align_scatter_kernel),
                        static_cast<int>(static_cast<size_t>(kAlignWarps) * MOE_MAX_EXPERTS * sizeof(int))))
    return MOE_ERR_CUDA;
  return launch_pdl(align_scatter_kernel, dim3(p.nchunks), dim3(kAlignThreads), smem, s, ids, num_pairs, E, p.chunk,
                    static_cast<const int32_t*>(chunk_base), done, sorted_ids, sorted_tok, topk > 0 ? topk : 1);
}

// Scratch for align run on the routing kernel's counts of T tokens: 256 bytes, then at most
// kSmallScan counts (rows of at least 4 tokens; align takes no more).
size_t align_tile_hist_bytes(int T, int E) {
  const long long n = std::min(static_cast<long long>((T + 3) / 4) * E, static_cast<long long>(kSmallScan));
  return 256 + align_up(static_cast<size_t>(n) * 4, 256);
}

// Whether the single-pass align can take tile_rows rows of pair_per_tile pairs instead of
// counting the pairs itself: every chunk is a whole number of rows, and the rows fit the
// single-pass scan.
bool align_takes_tile_hists(int num_pairs, int E, int tile_rows, int pairs_per_tile) {
  const AlignPlan p = align_plan(num_pairs);
  return pairs_per_tile > 0 && p.chunk % pairs_per_tile == 0 &&
         static_cast<long long>(tile_rows) * E <= kSmallScan && p.nchunks * E <= kSmallScan;
}

// Align with the first pass already done: tile_hist (in scratch, after its 256-byte
// header) holds tile_rows rows of per-expert counts of consecutive runs of
// pairs_per_tile pairs (the routing kernel's tiles). Also zeroes *zero_word.
moe_status_t launch_align_from_tile_hists(const int32_t* ids, int num_pairs, int E, int block_m,
                                          int32_t* sorted_ids, int32_t* expert_ids, int32_t* expert_offsets,
                                          int32_t* ntpp, const int32_t* tile_hist, int tile_rows,
                                          int pairs_per_tile, cudaStream_t s, int32_t* sorted_tok, int topk,
                                          int* zero_word) {
  const int cap = static_cast<int>(align_max_padded(num_pairs, E, block_m));
  const AlignPlan p = align_plan(num_pairs);
  const size_t smem = static_cast<size_t>(kAlignWarps + 3) * E * sizeof(int);
  if (!ensure_smem_attr(reinterpret_cast<const void*>(align_scan_scatter_kernel),
                        static_cast<int>(static_cast<size_t>(kAlignWarps + 3) * MOE_MAX_EXPERTS * sizeof(int))))
    return MOE_ERR_CUDA;
  return launch_pdl(align_scan_scatter_kernel, dim3(p.nchunks), dim3(kAlignThreads), smem, s, ids, num_pairs, E,
                    block_m, cap, p.chunk, p.nchunks, tile_hist, tile_rows, p.chunk / pairs_per_tile, sorted_ids,
                    sorted_tok, topk > 0 ? topk : 1, expert_ids, expert_offsets, ntpp, zero_word);
}

}  // namespace moe

extern "C" size_t moe_align_max_padded(int num_pairs, int E, int block_m) {
  return moe::align_max_padded(num_pairs, E, block_m);
}

extern "C" size_t moe_align_workspace_size(int num_pairs, int E, int block_m) {
  if (num_pairs < 0 || E < 1 || !moe::valid_block_m(block_m)) return 0;
  return moe::kWsHeader + moe::align_scratch_bytes(num_pairs, E);
}

extern "C" moe_status_t moe_align_block_size(const int32_t* topk_ids, int num_pairs, int E, int block_m,
                                             int32_t* sorted_token_ids, int32_t* expert_ids,
                                             int32_t* expert_offsets, int32_t* num_tokens_post_padded, void* ws,
                                             size_t ws_bytes, void* stream) {
  if (num_pairs < 0 || E < 1 || E > MOE_MAX_EXPERTS || !moe::valid_block_m(block_m)) return MOE_ERR_INVALID_ARG;
  const bool empty = moe::align_max_padded(num_pairs, E, block_m) == 0;
  if ((num_pairs > 0 && !topk_ids) || (!empty && (!sorted_token_ids || !expert_ids)) || !expert_offsets ||
      !num_tokens_post_padded)
    return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < moe_align_workspace_size(num_pairs, E, block_m) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  return moe::launch_align(topk_ids, num_pairs, E, block_m, sorted_token_ids, expert_ids, expert_offsets,
                           num_tokens_post_padded, w + moe::kWsHeader, reinterpret_cast<int*>(w),
                           moe::as_stream(stream), nullptr, 0, nullptr);
}
