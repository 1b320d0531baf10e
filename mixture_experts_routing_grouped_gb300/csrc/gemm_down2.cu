// down grouped GEMM + weighted combine on CTA pairs (tcgen05 cta_group::2).
//
// Follows the mini-sglang MoE chapter ("fused MoE", fused_moe_kernel and
// FusedMoeBackend.forward, second launch): for every row of the
// expert-sorted layout, o = h[row] @ W2[e]^T is scaled by the route weight of
// the row's pair and summed into the pair's token row of the fp32 accumulator.
//
// A cluster of two CTAs computes up to 256 rows (two consecutive 128-row blocks
// of one expert, block 2m + rank in CTA `rank`) x 256 columns of H per tile.
// Each CTA TMA-loads its own 128 rows of h (16 KB per 64-deep K step) and its
// half of the W2 tile (rows nt*256 + 128*rank + [0, 128), 16 KB); the even CTA
// issues one M=256 N=256 pair MMA per 16-deep K step. Every SM thus brings in
// 256 box rows per K step for 4.2 MFLOP of its own, against 384 for a one-SM
// 128 x 256 tile: tiled TMA moves about one 128-byte box row per 2.4 SM cycles,
// which made the one-SM down kernel load-bound. Each CTA keeps its 128 x 256
// accumulator double-buffered in tensor memory (512 columns), so the combine of
// one tile overlaps the main loop of the next.
//
// Kernel shape (one CTA per SM, 192 threads, clusters of 2): warps 0-3 epilogue
// (TMEM lane quarter = warp), warp 4 TMA producer, warp 5 owns the CTA's tensor
// memory and, in the even CTA, issues the MMAs.
//
// Cross-CTA protocol (all waits bounded; CTA-scope arrives and waits, since
// every operand arrives by TMA and is published by the barrier's byte count):
//   full[s]   (even CTA, 2 arrivals): one arrive.expect_tx per CTA for its bytes;
//   empty[s]  (both CTAs): one multicast commit after the MMAs of the slot;
//   tfull[b]  (both CTAs): one multicast commit after the last K step of a tile;
//   tempty[b] (even CTA, 8 arrivals): one per epilogue warp of either CTA.
#include "common.cuh"
#include "ptx.cuh"

#include <cuda.h>

namespace moe {

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);

namespace down2 {

constexpr int kRows = 128;
constexpr int kBN = 256;
constexpr int kHalfN = kBN / 2;
constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kABytes = kRows * kBK * 2;
constexpr int kBBytes = kHalfN * kBK * 2;
constexpr int kEpiWarps = 4;
constexpr int kTmaWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kTmemCols = 2 * kBN;
constexpr int kStagePitch = 36;
constexpr size_t kCtlBytes = 256 + 4 * (MOE_MAX_EXPERTS + 1) + 12 + kEpiWarps * 32 * kStagePitch * 4;
constexpr size_t kSmem = 1024 + kStages * (kABytes + kBBytes) + kCtlBytes;
static_assert(kSmem <= 232448, "shared memory per CTA");

struct DownArgs {
  const int32_t* sorted_ids;  // pair of each sorted row, num_pairs for padding
  const int32_t* sorted_tok;  // token of each sorted row, -1 for padding
  const int32_t* offsets;     // [E + 1] padded segment starts
  const float* topk_w;        // [num_pairs]
  float* y_acc;               // [T, H]
  int* err;
  int num_pairs, E;
  int K;                      // I
  int H;
  int n_tiles;                // H / 256
};

struct TileInfo {
  int e, row0, nblk, nt;
};

__device__ __forceinline__ TileInfo decode_tile(const int* pfx, const int32_t* __restrict__ offsets, int E,
                                               int n_tiles, int t) {
  const int mp = t / n_tiles;
  TileInfo ti;
  ti.nt = t - mp * n_tiles;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pfx[mid] <= mp) lo = mid; else hi = mid;
  }
  while (lo + 1 < E && pfx[lo + 1] <= mp) ++lo;
  ti.e = lo;
  const int local = mp - pfx[lo];
  const int b0 = __ldg(offsets + lo) / kRows + 2 * local;
  const int nb = (__ldg(offsets + lo + 1) - __ldg(offsets + lo)) / kRows;
  ti.row0 = b0 * kRows;
  ti.nblk = min(2, nb - 2 * local);
  return ti;
}

__global__ void __launch_bounds__(kThreads, 1)
    down_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                     const DownArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sA = raw_addr + pad;
  const uint32_t sB = sA + kStages * kABytes;
  uint8_t* ctl = smem + kStages * (kABytes + kBBytes);
  const uint32_t bar_base = ptx::smem_u32(ctl);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * (2 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * (2 * kStages + 2 + b); };
  const uint32_t done_bar = bar_base + 8u * (2 * kStages + 4);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl + 132);
  int* pfx = reinterpret_cast<int*>(ctl + 256);
  float* stg_all = reinterpret_cast<float*>(pfx + (MOE_MAX_EXPERTS + 1) + 3);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 2);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), 2 * kEpiWarps);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc_pair(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    ptx::tmem_relinquish_pair();
  } else if (warp == 1) {
    const int per = (args.E + 31) / 32;
    const int e0 = lane * per;
    int sum = 0;
    for (int j = 0; j < per; ++j) {
      const int e = e0 + j;
      if (e < args.E) {
        const int nb = (__ldg(args.offsets + e + 1) - __ldg(args.offsets + e)) / kRows;
        sum += (nb + 1) >> 1;
      }
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - sum;
    for (int j = 0; j < per; ++j) {
      const int e = e0 + j;
      if (e < args.E) {
        pfx[e] = run;
        const int nb = (__ldg(args.offsets + e + 1) - __ldg(args.offsets + e)) / kRows;
        run += (nb + 1) >> 1;
      }
    }
    if (lane == 31) pfx[args.E] = incl;
  } else if (warp == kTmaWarp && lane == 0) {
    ptx::prefetch_tmap(&map_a);
    ptx::prefetch_tmap(&map_b);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised before any remote arrive or multicast commit
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int tiles = pfx[args.E] * args.n_tiles;
  const int kblocks = args.K / kBK;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cid; t < tiles && ok; t += ncl) {
        const TileInfo ti = decode_tile(pfx, args.offsets, args.E, args.n_tiles, t);
        const bool present = static_cast<int>(rank) < ti.nblk;
        const int a_row = ti.row0 + static_cast<int>(rank) * kRows;
        const int b_row = ti.e * args.H + ti.nt * kBN + static_cast<int>(rank) * kHalfN;
        const uint32_t bytes = kBBytes + (present ? kABytes : 0);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t full_c = ptx::mapa_shared(full_bar(stage), 0);
          ptx::mbar_arrive_expect_tx_remote(full_c, bytes);
          if (present) ptx::tma_load_2d_pair(sA + stage * kABytes, &map_a, full_c, kb * kBK, a_row);
          ptx::tma_load_2d_pair(sB + stage * kBBytes, &map_b, full_c, kb * kBK, b_row);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (rank == 0 && ptx::elect_one()) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(2 * kRows, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = cid; t < tiles && ok; t += ncl, ++it) {
        const int b = it & 1;
        if (!ptx::mbar_wait(tempty_bar(b), ((static_cast<uint32_t>(it) >> 1) & 1u) ^ 1u, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t ad = ptx::sdesc_sw128(sA + stage * kABytes);
          const uint64_t bd = ptx::sdesc_sw128(sB + stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) ptx::mma_f16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          ptx::mma_commit_pair_mc(empty_bar(stage), 0x3);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) ptx::mma_commit_pair_mc(tfull_bar(b), 0x3);
      }
      ptx::mma_commit_pair_mc(done_bar, 0x1);
      ptx::mbar_wait_drain(done_bar, 0);
    }
    __syncwarp();
  } else {
    // Each warp drains its 32 accumulator rows 32 columns at a time through a
    // shared staging tile, so that one atomic instruction covers whole 128-byte
    // row segments of 4 rows.
    float* stg = stg_all + warp * 32 * kStagePitch;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    int it = 0;
    for (int t = cid; t < tiles; t += ncl, ++it) {
      const int b = it & 1;
      const TileInfo ti = decode_tile(pfx, args.offsets, args.E, args.n_tiles, t);
      const bool present = static_cast<int>(rank) < ti.nblk;
      int tok = -1;
      float w = 0.f;
      if (present) {
        const int pos = ti.row0 + static_cast<int>(rank) * kRows + warp * 32 + lane;
        tok = __ldg(args.sorted_tok + pos);
        if (tok >= 0) w = __ldg(args.topk_w + __ldg(args.sorted_ids + pos));
      }
      const bool ok = ptx::mbar_wait(tfull_bar(b), (static_cast<uint32_t>(it) >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      if (present) {
        const uint32_t tbase = tmem_base + lane_off + b * kBN;
        float* ybase = args.y_acc + ti.nt * kBN;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t d[32];
          ptx::tmem_ld32(tbase + c * 32, d);
          ptx::tmem_ld_wait();
          float4* srow = reinterpret_cast<float4*>(stg + lane * kStagePitch);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            srow[q] = make_float4(w * __uint_as_float(d[4 * q]), w * __uint_as_float(d[4 * q + 1]),
                                  w * __uint_as_float(d[4 * q + 2]), w * __uint_as_float(d[4 * q + 3]));
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = i * 4 + (lane >> 3);
            const int q = lane & 7;
            const int trow = __shfl_sync(0xffffffffu, tok, rl);
            const float4 v = reinterpret_cast<const float4*>(stg + rl * kStagePitch)[q];
            if (trow >= 0)
              atomicAdd(reinterpret_cast<float4*>(ybase + static_cast<size_t>(trow) * args.H + c * 32) + q, v);
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(ptx::mapa_shared(tempty_bar(b), 0));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still arrive on its barriers or read its smem
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  if (tid == 0 && *abort_flag) report_error(args.err, MOE_DEVERR_TIMEOUT);
}

int max_pair_grid() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms() & ~1), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, down_pair_kernel, &cfg) != cudaSuccess || clusters <= 0) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = 2 * std::min(clusters, num_sms() / 2);
  return cached[dev];
}

}  // namespace down2

bool down_pair2_supported(int H, int I) { return H % down2::kBN == 0 && I % down2::kBK == 0; }

moe_status_t launch_gemm_down_pair2(const __nv_bfloat16* h, const __nv_bfloat16* w2, const int32_t* sorted_ids,
                                    const int32_t* sorted_tok, const int32_t* offsets, const float* topk_w,
                                    float* y_acc, int* err, int num_pairs, int cap, int H, int I, int E,
                                    cudaStream_t s) {
  using namespace down2;
  if (!down_pair2_supported(H, I)) return MOE_ERR_UNSUPPORTED;
  CUtensorMap map_a, map_b;
  if (!make_tmap_bf16_2d(&map_a, h, static_cast<uint64_t>(cap), I)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&map_b, w2, static_cast<uint64_t>(E) * H, I)) return MOE_ERR_CUDA;
  DownArgs a{};
  a.sorted_ids = sorted_ids; a.sorted_tok = sorted_tok; a.offsets = offsets; a.topk_w = topk_w; a.y_acc = y_acc;
  a.err = err; a.num_pairs = num_pairs; a.E = E; a.K = I; a.H = H; a.n_tiles = H / kBN;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(down_pair_kernel), static_cast<int>(kSmem)))
    return MOE_ERR_CUDA;
  const int grid = max_pair_grid();
  if (grid < 2) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, down_pair_kernel, map_a, map_b, a) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace moe
