// moe_align_block_size: stable counting sort of the (token, expert) pairs by
// expert, each expert's segment padded to a multiple of block_m.
//
// Follows the mini-sglang MoE chapter ("fused MoE", moe_align_block_size):
// counts per expert, padded lengths, exclusive prefix sum, stable placement of
// every pair at seg_start[e] + rank-within-expert, sentinel num_pairs in the
// padding, the expert of every block.
//
// One CTA of 1024 threads. Warp w owns the contiguous pair range
// [w*S, (w+1)*S). Pass 1 counts the warp's pairs per expert into its own row of
// a shared [warp][expert] table (shared-memory atomics; counts do not depend on
// order). A block scan over experts turns the table into per-(warp, expert)
// write cursors. Pass 2 re-walks the range in order, 32 pairs at a time:
// __match_any_sync groups the lanes that carry the same expert, a pair's rank
// among them is the popcount of its lower peers, and it lands at cursor + rank.
// Walking the ranges in order makes the sort stable; no atomics decide
// positions. Ids are loaded kUnroll steps ahead so the loads overlap.
#include "common.cuh"

#include <algorithm>

namespace moe {
namespace {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kUnroll = 8;  // ids per lane loaded before they are used

__global__ void __launch_bounds__(kAlignThreads, 1)
    align_kernel(const int32_t* __restrict__ ids, int num_pairs, int E, int block_m, int cap,
                 int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                 int32_t* __restrict__ expert_offsets, int32_t* __restrict__ ntpp, int* __restrict__ err) {
  extern __shared__ int smem[];
  int* cur = smem;  // [kAlignWarps][E]: counts, then write cursors
  __shared__ int warp_tot[kAlignWarps];
  __shared__ int total_s;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) cur[i] = 0;
  __syncthreads();

  const int span = cdiv(num_pairs, kAlignWarps);
  const int lo = min(num_pairs, warp * span);
  const int hi = min(num_pairs, lo + span);

  // Pass 1: per-(warp, expert) counts; kUnroll ids per lane in flight.
  for (int b = lo; b < hi; b += 32 * kUnroll) {
    int e[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int p = b + j * 32 + lane;
      e[j] = (p < hi) ? __ldg(ids + p) : -1;
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int p = b + j * 32 + lane;
      if (p < hi) {
        if (e[j] < 0 || e[j] >= E) report_error(err, MOE_DEVERR_EXPERT_ID);
        else atomicAdd(&cur[warp * E + e[j]], 1);
      }
    }
  }
  __syncthreads();

  // Scan over experts (one expert per thread; E <= 1024).
  int count = 0, padded = 0;
  if (tid < E) {
    for (int w = 0; w < kAlignWarps; ++w) count += cur[w * E + tid];
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
    warp_tot[lane] = t;  // inclusive prefix over warps
    if (lane == 31) total_s = t;
  }
  __syncthreads();
  const int start = incl - padded + (warp > 0 ? warp_tot[warp - 1] : 0);
  const int total = total_s;
  if (tid < E) {
    expert_offsets[tid] = start;
    int c = start;
    for (int w = 0; w < kAlignWarps; ++w) {  // counts -> cursors
      const int n = cur[w * E + tid];
      cur[w * E + tid] = c;
      c += n;
    }
    for (int blk = start / block_m; blk < (start + padded) / block_m; ++blk) expert_ids[blk] = tid;
    for (int pos = start + count; pos < start + padded; ++pos) sorted_ids[pos] = num_pairs;
  }
  if (tid == 0) {
    expert_offsets[E] = total;
    *ntpp = total;
  }
  for (int pos = total + tid; pos < cap; pos += kAlignThreads) sorted_ids[pos] = num_pairs;
  for (int blk = total / block_m + tid; blk < cap / block_m; blk += kAlignThreads) expert_ids[blk] = -1;
  __syncthreads();

  // Pass 2: stable placement, walking the warp's range in order.
  for (int b = lo; b < hi; b += 32 * kUnroll) {
    int e[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int p = b + j * 32 + lane;
      const int v = (p < hi) ? __ldg(ids + p) : -1;
      e[j] = (v >= 0 && v < E) ? v : -1;
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int p = b + j * 32 + lane;
      const uint32_t peers = __match_any_sync(0xffffffffu, e[j]);
      int base = 0;
      if (e[j] >= 0) base = cur[warp * E + e[j]];
      __syncwarp();
      if (e[j] >= 0) {
        sorted_ids[base + __popc(peers & lt_mask)] = p;
        if ((peers & lt_mask) == 0) cur[warp * E + e[j]] = base + __popc(peers);
      }
      __syncwarp();
    }
  }
}

}  // namespace

size_t align_max_padded(int num_pairs, int E, int block_m) {
  if (num_pairs < 0 || E < 1 || block_m < 1) return 0;
  const size_t cap = static_cast<size_t>(num_pairs) + static_cast<size_t>(std::min(E, num_pairs)) * (block_m - 1);
  return align_up(cap, static_cast<size_t>(block_m));
}

bool valid_block_m(int bm) { return bm >= 1 && bm <= 256 && (bm & (bm - 1)) == 0; }

size_t align_smem_bytes(int E) { return static_cast<size_t>(kAlignWarps) * E * sizeof(int); }

moe_status_t launch_align(const int32_t* ids, int num_pairs, int E, int block_m, int32_t* sorted_ids,
                          int32_t* expert_ids, int32_t* expert_offsets, int32_t* ntpp, int* err, cudaStream_t s) {
  const int cap = static_cast<int>(align_max_padded(num_pairs, E, block_m));
  const size_t smem = align_smem_bytes(E);
  if (!ensure_smem_attr(reinterpret_cast<const void*>(align_kernel), static_cast<int>(align_smem_bytes(MOE_MAX_EXPERTS))))
    return MOE_ERR_CUDA;
  align_kernel<<<1, kAlignThreads, smem, s>>>(ids, num_pairs, E, block_m, cap, sorted_ids, expert_ids,
                                              expert_offsets, ntpp, err);
  return launch_status();
}

}  // namespace moe

extern "C" size_t moe_align_max_padded(int num_pairs, int E, int block_m) {
  return moe::align_max_padded(num_pairs, E, block_m);
}

extern "C" size_t moe_align_workspace_size(int num_pairs, int E, int block_m) {
  (void)num_pairs; (void)E; (void)block_m;
  return moe::kWsHeader;
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
  if (!ws || ws_bytes < moe_align_workspace_size(num_pairs, E, block_m)) return MOE_ERR_WORKSPACE;
  return moe::launch_align(topk_ids, num_pairs, E, block_m, sorted_token_ids, expert_ids, expert_offsets,
                           num_tokens_post_padded, static_cast<int*>(ws), moe::as_stream(stream));
}
