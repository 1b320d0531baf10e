// gate_up grouped GEMM on row-block pairs of the expert-sorted layout.
//
// Follows the mini-sglang MoE chapter ("fused MoE", fused_moe_kernel and
// FusedMoeBackend.forward): rows are the pairs sorted_token_ids[...] of one
// expert, gathered from X in-kernel (row pair / topk, read from the token
// table that the align step writes beside sorted_token_ids),
// C = X_rows @ W1[e]^T with the gate tile [n0, n0+128) stacked over the up
// tile [I+n0, I+n0+128), and the epilogue writes h = silu(gate)*up (the
// chapter's third exercise).
//
// Here a tile is up to two consecutive 128-row blocks of one expert (256 rows)
// x 256 accumulator columns: both row halves multiply the same staged weight
// tile, so each staged byte feeds 128 FLOP instead of 85 and the weights of an
// expert with two blocks are read once instead of twice. The two halves
// accumulate through two M=128 N=256 tcgen05.mma per K step into TMEM columns
// [0, 256) and [256, 512) (one accumulator set: the light SwiGLU epilogue is
// short next to the main loop). An expert with an odd number of blocks ends
// with a one-block tile.
//
// Tiles are handed out dynamically (the low-precision GMM article's dynamic
// task scheduling): a CTA starts on tile blockIdx.x and its TMA warp claims
// each further tile from an atomic counter (zeroed by the align step) a few K
// steps before the current tile's last weight load, then broadcasts the claimed
// id to the gather, MMA and epilogue warps through a 4-entry shared-memory
// queue. Tiles of two row blocks cost twice as much MMA work as an expert's odd
// last block; a fixed round-robin left the busiest SM about a fifth above the
// mean, claiming keeps every SM busy until the tiles run out. The claim order
// stays expert-major, so the CTAs in flight share an expert's weights and rows
// in L2.
//
// A K step is 32 columns (64-byte rows, 64B swizzle), so that the ring has
// seven (bf16, up to 256 experts) or six 32 KB slots: a slot's gathered rows and
// weight tile land 1-3 us after it is freed (L2 and HBM latency under load), and
// the slots keep five to six K steps of MMA work queued against that, where
// three 64-column slots left the MMA waiting for data for about 40 % of the kernel.
//
// The kernel is written in bytes of K: a K step is one 64-byte row segment of
// both operands, 32 bf16 or 64 FP8-e4m3 values, and either way two MMAs of 32
// bytes of K each (kind::f16 K=16, or kind::f8f6f4 K=32). The FP8 instance (the
// low-precision GMM article's layer: per-token activation scales, per-channel
// weight scales, fp32 accumulation, sections 2.3 and 4.3) gathers the rows of
// the per-token-quantised activations and multiplies each accumulator by its
// token's scale and its column's weight scale before the SwiGLU.
//
// Kernel shape (one persistent CTA per SM, 32 x (10 + slots) threads): warps 0-7
// epilogue (TMEM lane quarter = warp % 4, column chunks split between warps w and
// w+4, so that the single accumulator is drained -- and the next tile's MMAs
// start -- in half the time), warp 8 sends the weight tile of every ring slot by
// TMA, warps 9 .. 8+slots gather (warp 9+s fills both row halves of ring slot s),
// the last warp owns TMEM and issues the MMAs. A gather lane keeps the source offsets of its
// 32 rows of the tile in registers, so that its cp.async instructions issue
// back to back (reading each offset from shared memory between them made the
// gather issue-bound), and no gather lane waits for a TMA issue. The per-expert pair counts are prefix-summed in shared memory
// from expert_offsets at kernel start.
#include "common.cuh"
#include "ptx.cuh"

#include <cuda.h>

namespace moe {

bool make_tmap_bf16_2d_k32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);
bool make_tmap_u8_2d_k64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);

namespace pair {

constexpr int kHalf = 128;
constexpr int kBN = 256;
constexpr int kKBytes = 64;  // bytes of K per step: one 64-byte swizzle row (32 bf16 or 64 e4m3)
constexpr int kHalfBytes = kHalf * kKBytes;
constexpr int kABytes = 2 * kHalfBytes;
constexpr int kBBytes = kBN * kKBytes;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each draining half of the column chunks
constexpr int kTmaWarp = kEpiWarps;
constexpr int kGatherWarp0 = kEpiWarps + 1;
constexpr int kTmemCols = 2 * kBN;
constexpr int kQ = 4;                                        // claimed-tile queue entries
constexpr int kScaleFloats = 128;  // FP8: per epilogue warp, gate and up channel scales of its two column chunks
constexpr int kDeepMaxExperts = 256;  // the seven-slot instance's expert table holds this many experts

// One instance's ring depth and shared-memory layout. Seven slots (224 KB) leave room for
// an expert table of kDeepMaxExperts experts; six slots hold the full MOE_MAX_EXPERTS table
// and (FP8) the epilogue's channel scales.
template <bool F8, int S>
struct Shape {
  static constexpr int kStages = S;
  static constexpr int kMmaWarp = kGatherWarp0 + kStages;  // one gather warp per ring slot
  static constexpr int kThreads = 32 * (kMmaWarp + 1);
  static constexpr int kQConsumers = kStages + 1 + kEpiWarps;  // gather warps, MMA thread, epilogue warps
  static constexpr int kPfxCap = ((S == 7 ? kDeepMaxExperts : MOE_MAX_EXPERTS) + 1 + 3) & ~3;
  static constexpr size_t kCtlBytes = 320 + 4 * kPfxCap + (F8 ? kEpiWarps * kScaleFloats * 4 : 0);
  static constexpr size_t kSmem = 1024 + kStages * (kABytes + kBBytes) + kCtlBytes;
  static_assert(kSmem <= 232448, "gate_up shared memory exceeds the per-CTA maximum");
};

struct GemmArgs {
  const uint8_t* x;           // activations [T, K] (bf16, or e4m3 codes), K contiguous
  const float* sx;            // FP8: per-token activation scales [T]
  const float* sw;            // FP8: per-channel weight scales [E, 2I]
  const int32_t* sorted_tok;  // token of each sorted row, -1 for padding
  const int32_t* offsets;
  __nv_bfloat16* h;
  int* err;
  int E;
  int K;            // reduction length in elements
  int row_bytes;    // bytes of one activation row
  int I;
  int n_tiles;
  int b_rows_per_expert;
  float4* clear;    // fp32 accumulator of the down pass to zero (null: none)
  size_t clear_n4;  // its length in float4
  int* tile_counter;  // tiles claimed beyond the first gridDim.x (zero at launch); null: fixed round-robin
};

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

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
  const int b0 = __ldg(offsets + lo) / kHalf + 2 * local;
  const int nb = (__ldg(offsets + lo + 1) - __ldg(offsets + lo)) / kHalf;
  ti.row0 = b0 * kHalf;
  ti.nblk = min(2, nb - 2 * local);
  return ti;
}

template <bool F8, int S>
__global__ void __launch_bounds__(Shape<F8, S>::kThreads, 1)
    moe_gate_up_kernel(const __grid_constant__ CUtensorMap map_b, const GemmArgs args) {
  using Sh = Shape<F8, S>;
  constexpr int kStages = Sh::kStages;
  constexpr int kMmaWarp = Sh::kMmaWarp;
  constexpr int kQConsumers = Sh::kQConsumers;
  constexpr int kElemsPerStep = F8 ? kKBytes : kKBytes / 2;  // K elements per step
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
  auto qfull_bar = [&](int q) { return bar_base + 8u * (2 * kStages + 3 + q); };
  auto qempty_bar = [&](int q) { return bar_base + 8u * (2 * kStages + 3 + kQ + q); };
  static_assert(8 * (2 * kStages + 3 + 2 * kQ) <= 256, "barriers overlap the control words");
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl + 260);
  volatile int* tq = reinterpret_cast<volatile int*>(ctl + 272);  // [kQ] claimed tile ids
  int* pfx = reinterpret_cast<int*>(ctl + 320);                   // [E + 1], E + 1 <= Sh::kPfxCap
  float* scl_all = reinterpret_cast<float*>(pfx + Sh::kPfxCap);   // FP8: [kEpiWarps][kScaleFloats]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 2);  // weight expect_tx arrive + the slot's gather warp
      ptx::mbar_init(empty_bar(s), 1);
    }
    ptx::mbar_init(tfull_bar, 1);
    ptx::mbar_init(tempty_bar, 32 * kEpiWarps);
    ptx::mbar_init(done_bar, 1);
    for (int q = 0; q < kQ; ++q) {
      ptx::mbar_init(qfull_bar(q), 1);
      ptx::mbar_init(qempty_bar(q), kQConsumers);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    ptx::tmem_relinquish();
  } else if (warp == kTmaWarp) {
    ptx::prefetch_tmap(&map_b);
  }
  pdl_wait();  // from here on: reads of what the kernels before this one wrote
  if (warp == 1) {
    const int per = (args.E + 31) / 32;
    const int e0 = lane * per;
    int sum = 0;
    for (int j = 0; j < per; ++j) {
      const int e = e0 + j;
      if (e < args.E) {
        const int nb = (__ldg(args.offsets + e + 1) - __ldg(args.offsets + e)) / kHalf;
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
        const int nb = (__ldg(args.offsets + e + 1) - __ldg(args.offsets + e)) / kHalf;
        run += (nb + 1) >> 1;
      }
    }
    if (lane == 31) pfx[args.E] = incl;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int tiles = pfx[args.E] * args.n_tiles;
  const int kblocks = args.K / kElemsPerStep;  // >= 1 (the host requires whole 64-byte steps)
  // The next tile is claimed, and read by the gather warps for their token
  // prefetch, from this K step of the current tile on.
  const int claim_at = kblocks > 2 * kStages ? kblocks - 2 * kStages : 0;

  // Queue entry j (the CTA's j-th tile): read once by every consumer warp (all
  // its lanes, warp_wide) or by the single MMA thread.
  auto read_tile = [&](int j, int& t_out, bool warp_wide) -> bool {
    const int q = j % kQ;
    bool ok = ptx::mbar_wait(qfull_bar(q), static_cast<uint32_t>(j / kQ) & 1u, abort_flag);
    if (warp_wide) ok = __all_sync(0xffffffffu, ok);  // the warp goes on, or leaves, as one
    t_out = ok ? tq[q] : tiles;
    if (warp_wide) __syncwarp();
    if (ok && (!warp_wide || lane == 0)) ptx::mbar_arrive(qempty_bar(q));
    return ok;
  };

  if (warp == kTmaWarp) {
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      auto publish = [&](int j, int t) -> bool {
        const int q = j % kQ;
        if (!ptx::mbar_wait(qempty_bar(q), (static_cast<uint32_t>(j / kQ) & 1u) ^ 1u, abort_flag)) return false;
        tq[q] = t;
        ptx::mbar_arrive(qfull_bar(q));  // release: the id is visible to the waiting consumers
        return true;
      };
      int t = blockIdx.x;
      bool ok = publish(0, t);
      for (int j = 0; ok && t < tiles; ++j) {
        const TileInfo ti = decode_tile(pfx, args.offsets, args.E, args.n_tiles, t);
        const int b_row0 = ti.e * args.b_rows_per_expert + ti.nt * kHalf;
        int t_next = tiles;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (kb == claim_at) {
            t_next = args.tile_counter ? static_cast<int>(gridDim.x) + atomicAdd(args.tile_counter, 1)
                                       : t + static_cast<int>(gridDim.x);
            if (!publish(j + 1, t_next)) { ok = false; break; }
          }
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t b_dst = sB + stage * kBBytes;
          ptx::mbar_arrive_expect_tx(full_bar(stage), kBBytes);
          ptx::tma_load_2d(b_dst, &map_b, full_bar(stage), kb * kElemsPerStep, b_row0);
          ptx::tma_load_2d(b_dst + kBBytes / 2, &map_b, full_bar(stage), kb * kElemsPerStep, b_row0 + args.I);
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        t = t_next;
      }
#pragma unroll
      for (int st = 0; st < kStages; ++st) {
        const int fills = issued / kStages + (st < issued % kStages ? 1 : 0);
        if (fills > 0) ptx::mbar_wait_drain(full_bar(st), (fills - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp >= kGatherWarp0 && warp < kMmaWarp) {
    const int slot = warp - kGatherWarp0;
    const uint32_t a_dst = sA + slot * kABytes;
    const int chunk = lane & 3;  // 16-byte chunk of a 64-byte row
    const int rsub = lane >> 2;  // row within an 8-row group
    const uint8_t* xc = args.x + chunk * 16;
    // Rows 8i + rsub of the tile (i < 16: first block, i >= 16: second): offs
    // holds the current tile's source offsets, pre the next tile's tokens,
    // loaded while this tile streams.
    constexpr int kRows = 2 * kHalf / 8;
    int offs[kRows], pre[kRows];
    int cur_j = -1, pre_j = -1, pre_t = tiles;
    int nblk = 0, pre_nblk = 0;
    // Reads queue entry jj and loads that tile's token rows into pre[].
    auto fetch = [&](int jj) -> bool {
      int tt;
      if (!read_tile(jj, tt, true)) return false;
      pre_j = jj;
      pre_t = tt;
      pre_nblk = 0;
      if (tt < tiles) {
        const TileInfo tj = decode_tile(pfx, args.offsets, args.E, args.n_tiles, tt);
        pre_nblk = tj.nblk;
        const int32_t* toks = args.sorted_tok + tj.row0 + rsub;
#pragma unroll
        for (int i = 0; i < kRows; ++i) pre[i] = (i < kRows / 2 || tj.nblk == 2) ? __ldg(toks + 8 * i) : -1;
      }
      return true;
    };
    // The warp reads the queue entries in order, each exactly once: at its first
    // K step of tile j it reads any entries up to j that it has not read yet
    // (tiles in which it has no K step when a tile has fewer K steps than the
    // ring has slots), and it stops at the first entry past the last tile. When
    // tiles have kblocks >= kStages steps it has a step in every tile and in
    // every tile's last 2 * kStages steps, so the next tile's tokens are
    // prefetched while the current one streams.
    for (int g = slot;; g += kStages) {
      const int j = g / kblocks;
      const int kb = g - j * kblocks;
      if (j != cur_j) {
        // never read past the entry that ends the tiles: nothing is published after it
        bool aborted = false;
        while (pre_j < j && !(pre_j >= 0 && pre_t >= tiles)) {
          if (!fetch(pre_j + 1)) { aborted = true; break; }
        }
        if (aborted || pre_t >= tiles) break;
        cur_j = j;
        nblk = pre_nblk;
#pragma unroll
        for (int i = 0; i < kRows; ++i) offs[i] = pre[i] >= 0 ? pre[i] * args.row_bytes : -1;
      }
      if (kb >= claim_at && pre_j == j && !fetch(j + 1)) break;
      const uint32_t use = static_cast<uint32_t>(g / kStages);
      const bool ok = ptx::mbar_wait(empty_bar(slot), (use & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      {
        const int k0 = kb * kKBytes;
        // 64B swizzle: chunk c of row r at r * 64 + ((c ^ ((r >> 1) & 3)) << 4)
#pragma unroll
        for (int i = 0; i < kRows / 2; ++i) {
          const int r = i * 8 + rsub;
          const int off = offs[i];
          const uint32_t dst = a_dst + r * 64 + ((chunk ^ ((r >> 1) & 3)) << 4);
          ptx::cp_async_16(dst, off >= 0 ? xc + off + k0 : args.x, off >= 0 ? 16u : 0u);
        }
        if (nblk == 2) {
#pragma unroll
          for (int i = kRows / 2; i < kRows; ++i) {
            const int r = i * 8 + rsub;
            const int off = offs[i];
            const uint32_t dst = a_dst + r * 64 + ((chunk ^ ((r >> 1) & 3)) << 4);
            ptx::cp_async_16(dst, off >= 0 ? xc + off + k0 : args.x, off >= 0 ? 16u : 0u);
          }
        }
        ptx::cp_async_commit();
        ptx::cp_async_wait<0>();
        ptx::fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(full_bar(slot));
    }
    ptx::cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    if (ptx::elect_one()) {
      constexpr uint32_t idesc = F8 ? ptx::idesc_e4m3_f32(kHalf, kBN) : ptx::idesc_bf16_f32(kHalf, kBN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int t;
        if (!read_tile(it, t, false) || t >= tiles) break;
        const TileInfo ti = decode_tile(pfx, args.offsets, args.E, args.n_tiles, t);
        if (!ptx::mbar_wait(tempty_bar, (static_cast<uint32_t>(it) & 1u) ^ 1u, abort_flag)) break;
        ptx::tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t a0 = ptx::sdesc_sw64(sA + stage * kABytes);
          const uint64_t a1 = ptx::sdesc_sw64(sA + stage * kABytes + kHalfBytes);
          const uint64_t bd = ptx::sdesc_sw64(sB + stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kKBytes / 32; ++kk) {  // 32 bytes of K per MMA
            if constexpr (F8) {
              ptx::mma_f8(tmem_base, a0 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
              if (ti.nblk == 2) ptx::mma_f8(tmem_base + kBN, a1 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
            } else {
              ptx::mma_f16(tmem_base, a0 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
              if (ti.nblk == 2) ptx::mma_f16(tmem_base + kBN, a1 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
            }
          }
          ptx::mma_commit(empty_bar(stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) ptx::mma_commit(tfull_bar);
      }
      ptx::mma_commit(done_bar);
      ptx::mbar_wait_drain(done_bar, 0);
    }
    __syncwarp();
  } else {
    float* scl = scl_all + warp * kScaleFloats;  // FP8: [chunk 0..1][gate 32 | up 32]
    const int quarter = warp & 3;       // TMEM lane quarter (rows 32*quarter ..)
    const int cpart = warp >> 2;        // column chunks [2*cpart, 2*cpart + 2) of each row half
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    if (args.clear) {
      // Zero this CTA's share of the down pass's accumulator while the first
      // tile's main loop runs (the down kernel starts after this kernel ends).
      const size_t per = (args.clear_n4 + gridDim.x - 1) / gridDim.x;
      const size_t lo = per * blockIdx.x;
      const size_t hi = lo + per < args.clear_n4 ? lo + per : args.clear_n4;
      // evict-last: the zeroed rows stay in L2 through this kernel's weight stream
      // until the down kernel reduces into them
      const uint64_t pol = ptx::l2_policy_evict_last();
      for (size_t i = lo + tid; i < hi; i += 32 * kEpiWarps)
        ptx::st_f32x4(reinterpret_cast<float*>(args.clear + i), make_float4(0.f, 0.f, 0.f, 0.f), pol);
    }
    for (int it = 0;; ++it) {
      int t;
      if (!read_tile(it, t, true) || t >= tiles) break;
      const TileInfo ti = decode_tile(pfx, args.offsets, args.E, args.n_tiles, t);
      const int n0 = ti.nt * kHalf;
      // FP8: while the tile's MMAs run, fetch the token scale of this lane's row in
      // each row half and stage the warp's 128 channel scales in shared memory, so
      // that no global load sits between the accumulator and the SwiGLU.
      float rs_half[2] = {1.f, 1.f};
      if constexpr (F8) {
        const int cl = lane >> 4, part = (lane >> 3) & 1, q = lane & 7;
        const float* src =
            args.sw + static_cast<size_t>(ti.e) * 2 * args.I + part * args.I + n0 + (2 * cpart + cl) * 32 + q * 4;
        reinterpret_cast<float4*>(scl)[lane] = __ldg(reinterpret_cast<const float4*>(src));
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int tok = hb < ti.nblk ? __ldg(args.sorted_tok + ti.row0 + hb * kHalf + quarter * 32 + lane) : -1;
          rs_half[hb] = tok >= 0 ? __ldg(args.sx + tok) : 0.f;  // 0 for padding rows
        }
        __syncwarp();
      }
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(tfull_bar, static_cast<uint32_t>(it) & 1u, abort_flag))) break;
      ptx::tc_fence_after();
      for (int half = 0; half < ti.nblk; ++half) {
        const uint32_t tbase = tmem_base + lane_off + half * kBN;
        const int rowbase = ti.row0 + half * kHalf + quarter * 32;
        const float rs = rs_half[half];
#pragma unroll 1
        for (int c = 2 * cpart; c < 2 * cpart + 2; ++c) {
          uint32_t g[32], u[32];
          ptx::tmem_ld32(tbase + c * 32, g);
          ptx::tmem_ld32(tbase + kHalf + c * 32, u);
          ptx::tmem_ld_wait();
          if constexpr (F8) {
            // g = sx[token] * sw[e, n] * acc_g, u = sx[token] * sw[e, I + n] * acc_u
            const float4* swg = reinterpret_cast<const float4*>(scl + (c - 2 * cpart) * 64);
            const float4* swu = swg + 8;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 a = swg[j / 4];
              const float4 b = swu[j / 4];
              g[j] = __float_as_uint(rs * a.x * __uint_as_float(g[j]));
              g[j + 1] = __float_as_uint(rs * a.y * __uint_as_float(g[j + 1]));
              g[j + 2] = __float_as_uint(rs * a.z * __uint_as_float(g[j + 2]));
              g[j + 3] = __float_as_uint(rs * a.w * __uint_as_float(g[j + 3]));
              u[j] = __float_as_uint(rs * b.x * __uint_as_float(u[j]));
              u[j + 1] = __float_as_uint(rs * b.y * __uint_as_float(u[j + 1]));
              u[j + 2] = __float_as_uint(rs * b.z * __uint_as_float(u[j + 2]));
              u[j + 3] = __float_as_uint(rs * b.w * __uint_as_float(u[j + 3]));
            }
          }
          uint32_t hw[16];  // this lane's row: h columns c*32 .. c*32+31 as bf16 pairs
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
            const float h1 = silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
            const __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
            hw[j] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          // Lanes 2i and 2i+1 swap halves (one shuffle a word), so that each 32-byte store of
          // a lane pair covers the 64 bytes of one row: a store instruction writes 16 whole
          // row segments. Storing each lane's own row instead (32 rows an instruction) took
          // the kernel 3 % longer, and staging through shared memory leaves no room for a
          // seventh ring slot.
          const bool odd = (lane & 1) != 0;
          uint32_t lo[8], hi[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? hw[k] : hw[8 + k], 1);
            lo[k] = odd ? got : hw[k];      // row 2i, columns [16 odd, +16)
            hi[k] = odd ? hw[8 + k] : got;  // row 2i+1, same columns
          }
          __nv_bfloat16* dst =
              args.h + static_cast<size_t>(rowbase + (lane & ~1)) * args.I + n0 + c * 32 + (odd ? 16 : 0);
          ptx::st_b32x8(dst, lo);
          ptx::st_b32x8(dst + args.I, hi);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty_bar);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem_base, kTmemCols);
  if (tid == 0 && *abort_flag) report_error(args.err, MOE_DEVERR_TIMEOUT);
}

}  // namespace pair

namespace {

template <bool F8, int S>
moe_status_t launch_gate_up_shape(const CUtensorMap& map_b, const pair::GemmArgs& a, cudaStream_t s) {
  using Sh = pair::Shape<F8, S>;
  if (a.E + 1 > Sh::kPfxCap) return MOE_ERR_UNSUPPORTED;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(pair::moe_gate_up_kernel<F8, S>), static_cast<int>(Sh::kSmem)))
    return MOE_ERR_CUDA;
  return launch_pdl(pair::moe_gate_up_kernel<F8, S>, dim3(num_sms()), dim3(Sh::kThreads), Sh::kSmem, s, map_b, a);
}

// bf16: seven ring slots up to kDeepMaxExperts experts, six beyond (the full expert table
// takes the seventh slot's room). The MMA waits on its operands' latency, so a deeper ring
// runs faster: 210, 199 and 191 us with five, six and seven slots at T=4096, H=2048,
// I=768, E=128, top-8. FP8 keeps six slots: its channel scales take the room of the seventh.
template <bool F8>
moe_status_t launch_gate_up(const CUtensorMap& map_b, const pair::GemmArgs& a, cudaStream_t s) {
  if (!F8 && a.E <= pair::kDeepMaxExperts) return launch_gate_up_shape<false, 7>(map_b, a, s);
  return launch_gate_up_shape<F8, 6>(map_b, a, s);
}

}  // namespace

moe_status_t launch_gemm_gate_up_pairs(const __nv_bfloat16* x, const __nv_bfloat16* w1, const int32_t* sorted_tok,
                                       const int32_t* offsets, __nv_bfloat16* h, int* err, int num_pairs, int topk,
                                       int H, int I, int E, float* y_clear, size_t y_clear_floats,
                                       int* tile_counter, cudaStream_t s) {
  (void)num_pairs; (void)topk;
  using namespace pair;
  if ((H * 2) % kKBytes != 0) return MOE_ERR_UNSUPPORTED;
  CUtensorMap map_b;
  if (!make_tmap_bf16_2d_k32(&map_b, w1, static_cast<uint64_t>(E) * 2 * I, H)) return MOE_ERR_CUDA;
  GemmArgs a{};
  a.x = reinterpret_cast<const uint8_t*>(x); a.sorted_tok = sorted_tok; a.offsets = offsets; a.h = h; a.err = err;
  a.E = E; a.K = H; a.row_bytes = H * 2; a.I = I;
  a.n_tiles = I / kHalf; a.b_rows_per_expert = 2 * I;
  a.clear = reinterpret_cast<float4*>(y_clear); a.clear_n4 = y_clear ? y_clear_floats / 4 : 0;
  a.tile_counter = tile_counter;
  return launch_gate_up<false>(map_b, a, s);
}

moe_status_t launch_gemm_gate_up_pairs_fp8(const uint8_t* qx, const float* sx, const uint8_t* w1, const float* sw1,
                                           const int32_t* sorted_tok, const int32_t* offsets, __nv_bfloat16* h,
                                           int* err, int H, int I, int E, float* y_clear, size_t y_clear_floats,
                                           int* tile_counter, cudaStream_t s) {
  using namespace pair;
  if (H % kKBytes != 0) return MOE_ERR_UNSUPPORTED;
  CUtensorMap map_b;
  if (!make_tmap_u8_2d_k64(&map_b, w1, static_cast<uint64_t>(E) * 2 * I, H)) return MOE_ERR_CUDA;
  GemmArgs a{};
  a.x = qx; a.sx = sx; a.sw = sw1; a.sorted_tok = sorted_tok; a.offsets = offsets; a.h = h; a.err = err;
  a.E = E; a.K = H; a.row_bytes = H; a.I = I;
  a.n_tiles = I / kHalf; a.b_rows_per_expert = 2 * I;
  a.clear = reinterpret_cast<float4*>(y_clear); a.clear_n4 = y_clear ? y_clear_floats / 4 : 0;
  a.tile_counter = tile_counter;
  return launch_gate_up<true>(map_b, a, s);
}

}  // namespace moe
