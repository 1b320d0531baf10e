// gate_up grouped GEMM on CTA pairs (two SMs per tile, tcgen05 cta_group::2).
//
// Same computation as the one-SM kernels (the mini-sglang MoE chapter, "fused
// MoE": fused_moe_kernel and FusedMoeBackend.forward): the rows of a tile are
// pairs sorted_token_ids[...] of one expert, gathered from X in-kernel (row
// pair / topk, read from the align step's token table), C = X_rows @ W1[e]^T,
// and the epilogue writes
// h = silu(gate) * up (the chapter's third exercise).
//
// A cluster of two CTAs computes up to 256 rows (two consecutive 128-row blocks
// of one expert: block 2m + rank in CTA `rank`) x 512 accumulator columns: the
// gate columns [n0, n0 + 256) in tensor-memory columns [0, 256) and the up
// columns [I + n0, I + n0 + 256) in [256, 512). Every 64-deep K step is two
// M=256 N=256 pair MMAs issued by the even CTA; each CTA gathers only its own
// 128 rows of X (cp.async, 16 KB) and loads its half of both weight tiles by TMA
// (W1 rows n0 + 128*rank + [0, 128) of the gate and of the up block, 32 KB), so
// one SM stages 48 KB per 8.4 MFLOP of which 16 KB is gathered. A one-SM tile of
// the same work stages 64 KB with 32 KB gathered, and the per-lane gather is
// the slowest path into shared memory (about 29 GB/s per SM against about
// 100 GB/s per SM for tiled TMA loads from L2), so halving it is what the pair
// buys; the smaller stage also makes room for a fourth ring slot.
//
// Kernel shape (one CTA per SM, 320 threads, clusters of 2): warps 0-3 epilogue
// (TMEM lane quarter = warp), warp 4 sends the weight halves of every ring slot
// by TMA, warps 5-8 gather (warp 5+s owns ring slot s), warp 9 owns the CTA's
// tensor memory and, in the even CTA, issues the MMAs. A gather lane keeps the
// source offsets of its 32 rows of the tile in registers, so that its cp.async
// instructions issue back to back (each one waiting for a shared-memory load of
// its row offset made the gather issue-bound), and no gather lane ever waits for
// a TMA issue.
//
// Cross-CTA protocol (all waits bounded). Barrier operations are CTA-scope
// except where the odd CTA's gathered rows (generic-proxy writes to its own
// shared memory, read by the even CTA's MMA) are published: that arrive is a
// cluster-scope release and the MMA's wait on full[s] a cluster-scope acquire.
// Cluster-scope operations on every ring step cost several times the step.
//   full[s]  (even CTA, 4 arrivals): per CTA one arrive.expect_tx of its weight
//            bytes (completed by its TMA loads) and one arrive after its gather;
//   empty[s] (both CTAs): one multicast commit after the MMAs of the slot;
//   tfull    (both CTAs): one multicast commit after the last K step of a tile;
//   tempty   (even CTA, 8 arrivals): one per epilogue warp of either CTA.
#include "common.cuh"
#include "ptx.cuh"

#include <cuda.h>

namespace moe {

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);

namespace pair2 {

constexpr int kRows = 128;
constexpr int kBN = 256;
constexpr int kHalfN = kBN / 2;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kRows * kBK * 2;
constexpr int kBHalfBytes = kHalfN * kBK * 2;
constexpr int kBBytes = 2 * kBHalfBytes;
constexpr int kEpiWarps = 4;
constexpr int kTmaWarp = kEpiWarps;
constexpr int kGatherWarp0 = kEpiWarps + 1;
constexpr int kMmaWarp = kGatherWarp0 + kStages;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kTmemCols = 2 * kBN;
constexpr int kStagePitch = 36;
constexpr size_t kCtlBytes = 256 + 4 * (MOE_MAX_EXPERTS + 1) + 12 + kEpiWarps * 32 * kStagePitch * 4;
constexpr size_t kSmem = 1024 + kStages * (kABytes + kBBytes) + kCtlBytes;
static_assert(kSmem <= 232448, "shared memory per CTA");

struct GemmArgs {
  const __nv_bfloat16* x;
  const int32_t* sorted_tok;  // token of each sorted row, -1 for padding
  const int32_t* offsets;
  __nv_bfloat16* h;
  int* err;
  int E;
  int K;
  int I;
  int n_tiles;
};

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

struct TileInfo {
  int e, row0, nblk, nt;
};

// Tile t = (row-block pair m, n-tile nt) in expert-major order; pfx[e] is the
// first pair index of expert e.
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
    gate_up_pair_kernel(const __grid_constant__ CUtensorMap map_b, const GemmArgs args) {
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
  const uint32_t tfull_bar = bar_base + 8u * (2 * kStages);
  const uint32_t tempty_bar = bar_base + 8u * (2 * kStages + 1);
  const uint32_t done_bar = bar_base + 8u * (2 * kStages + 2);
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
      ptx::mbar_init(full_bar(s), 4);
      ptx::mbar_init(empty_bar(s), 1);
    }
    ptx::mbar_init(tfull_bar, 1);
    ptx::mbar_init(tempty_bar, 2 * kEpiWarps);
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
  } else if (warp == kTmaWarp) {
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
    // Weight halves of every K step, in ring order.
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = cid; t < tiles && ok; t += ncl) {
      const TileInfo ti = decode_tile(pfx, args.offsets, args.E, args.n_tiles, t);
      const int b_row0 = ti.e * 2 * args.I + ti.nt * kBN + static_cast<int>(rank) * kHalfN;
      for (int kb = 0; kb < kblocks; ++kb) {
        const bool w = ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t b_dst = sB + stage * kBBytes;
          const uint32_t full_c = ptx::mapa_shared(full_bar(stage), 0);
          ptx::mbar_arrive_expect_tx_remote(full_c, kBBytes);
          ptx::tma_load_2d_pair(b_dst, &map_b, full_c, kb * kBK, b_row0);
          ptx::tma_load_2d_pair(b_dst + kBHalfBytes, &map_b, full_c, kb * kBK, b_row0 + args.I);
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp >= kGatherWarp0 && warp < kMmaWarp) {
    // Rows of X for ring slot `slot`: lane (rsub, chunk) copies 16-byte chunk
    // `chunk` of rows 4i + rsub, i < 32, of this CTA's 128-row block.
    const int slot = warp - kGatherWarp0;
    const uint32_t full_c = ptx::mapa_shared(full_bar(slot), 0);
    const uint32_t a_dst = sA + slot * kABytes;
    const int chunk = lane & 7;
    const int rsub = lane >> 3;
    const __nv_bfloat16* xc = args.x + chunk * 8;
    // offs: source offsets of the current tile's rows; pre: the next tile's
    // tokens, loaded while this tile streams.
    int offs[kRows / 4], pre[kRows / 4];
    int cached_t = -1, pre_t = -1;
    bool present = false, pre_present = false;
    auto load_toks = [&](int tt) {
      const TileInfo tj = decode_tile(pfx, args.offsets, args.E, args.n_tiles, tt);
      pre_present = static_cast<int>(rank) < tj.nblk;
      const int32_t* toks = args.sorted_tok + tj.row0 + static_cast<int>(rank) * kRows + rsub;
#pragma unroll
      for (int i = 0; i < kRows / 4; ++i) pre[i] = pre_present ? __ldg(toks + 4 * i) : -1;
      pre_t = tt;
    };
    for (int g = slot;; g += kStages) {
      const int t_local = g / kblocks;
      const int t = cid + t_local * ncl;
      if (t >= tiles) break;
      const int kb = g - t_local * kblocks;
      if (t != cached_t) {
        if (pre_t != t) load_toks(t);
        present = pre_present;
#pragma unroll
        for (int i = 0; i < kRows / 4; ++i) offs[i] = pre[i] >= 0 ? pre[i] * args.K : -1;
        cached_t = t;
        if (t + ncl < tiles) load_toks(t + ncl);
      }
      const uint32_t use = static_cast<uint32_t>(g / kStages);
      const bool ok = ptx::mbar_wait(empty_bar(slot), (use & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (present) {
        const int k0 = kb * kBK;
#pragma unroll
        for (int i = 0; i < kRows / 4; ++i) {
          const int r = i * 4 + rsub;
          const uint32_t dst = a_dst + r * 128 + ((chunk ^ (r & 7)) << 4);
          const int off = offs[i];
          ptx::cp_async_16(dst, off >= 0 ? xc + off + k0 : args.x, off >= 0 ? 16u : 0u);
        }
        ptx::cp_async_commit();
        ptx::cp_async_wait<0>();
        ptx::fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) ptx::mbar_arrive(full_bar(slot));
        else ptx::mbar_arrive_cluster(full_c);
      }
    }
    ptx::cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    if (rank == 0 && ptx::elect_one()) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(2 * kRows, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = cid; t < tiles && ok; t += ncl, ++it) {
        if (!ptx::mbar_wait(tempty_bar, (static_cast<uint32_t>(it) & 1u) ^ 1u, abort_flag)) break;
        ptx::tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait_cluster(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t ad = ptx::sdesc_sw128(sA + stage * kABytes);
          const uint64_t bg = ptx::sdesc_sw128(sB + stage * kBBytes);
          const uint64_t bu = ptx::sdesc_sw128(sB + stage * kBBytes + kBHalfBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            ptx::mma_f16_pair(tmem_base, ad + 2 * kk, bg + 2 * kk, idesc, (kb | kk) != 0);
            ptx::mma_f16_pair(tmem_base + kBN, ad + 2 * kk, bu + 2 * kk, idesc, (kb | kk) != 0);
          }
          ptx::mma_commit_pair_mc(empty_bar(stage), 0x3);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) ptx::mma_commit_pair_mc(tfull_bar, 0x3);
      }
      ptx::mma_commit_pair_mc(done_bar, 0x1);
      ptx::mbar_wait_drain(done_bar, 0);
    }
    __syncwarp();
  } else {
    float* stg = stg_all + warp * 32 * kStagePitch;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tempty_c = ptx::mapa_shared(tempty_bar, 0);
    int it = 0;
    for (int t = cid; t < tiles; t += ncl, ++it) {
      const TileInfo ti = decode_tile(pfx, args.offsets, args.E, args.n_tiles, t);
      const bool ok = ptx::mbar_wait(tfull_bar, static_cast<uint32_t>(it) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      if (static_cast<int>(rank) < ti.nblk) {
        const uint32_t tbase = tmem_base + lane_off;
        const int rowbase = ti.row0 + static_cast<int>(rank) * kRows + warp * 32;
        const int n0 = ti.nt * kBN;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t g[32], u[32];
          ptx::tmem_ld32(tbase + c * 32, g);
          ptx::tmem_ld32(tbase + kBN + c * 32, u);
          ptx::tmem_ld_wait();
          uint32_t* srow = reinterpret_cast<uint32_t*>(stg + lane * kStagePitch);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
            const float h1 = silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
            const __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
            srow[j] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = i * 4 + (lane >> 3);
            const int q = lane & 7;
            const uint32_t* src = reinterpret_cast<const uint32_t*>(stg + rl * kStagePitch) + 2 * q;
            uint2* dst =
                reinterpret_cast<uint2*>(args.h + static_cast<size_t>(rowbase + rl) * args.I + n0 + c * 32) + q;
            *dst = make_uint2(src[0], src[1]);
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(tempty_c);
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
  if (cudaOccupancyMaxActiveClusters(&clusters, gate_up_pair_kernel, &cfg) != cudaSuccess || clusters <= 0) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = 2 * std::min(clusters, num_sms() / 2);
  return cached[dev];
}

}  // namespace pair2

bool gate_up_pair2_supported(int I) { return I % pair2::kBN == 0; }

moe_status_t launch_gemm_gate_up_pair2(const __nv_bfloat16* x, const __nv_bfloat16* w1, const int32_t* sorted_tok,
                                       const int32_t* offsets, __nv_bfloat16* h, int* err, int num_pairs, int topk,
                                       int H, int I, int E, cudaStream_t s) {
  using namespace pair2;
  (void)num_pairs; (void)topk;
  if (!gate_up_pair2_supported(I)) return MOE_ERR_UNSUPPORTED;
  CUtensorMap map_b;
  if (!make_tmap_bf16_2d(&map_b, w1, static_cast<uint64_t>(E) * 2 * I, H)) return MOE_ERR_CUDA;
  GemmArgs a{};
  a.x = x; a.sorted_tok = sorted_tok; a.offsets = offsets; a.h = h; a.err = err;
  a.E = E; a.K = H; a.I = I;
  a.n_tiles = I / kBN;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(gate_up_pair_kernel), static_cast<int>(kSmem)))
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
  if (cudaLaunchKernelEx(&cfg, gate_up_pair_kernel, map_b, a) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace moe
