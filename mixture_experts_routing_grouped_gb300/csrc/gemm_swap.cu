// Swap-AB grouped GEMMs of the MoE layer: weight rows on the MMA's M side,
// an expert's tokens on its N side.
//
// Follows the vLLM fused-MoE article (spke.com), "Swap-AB": when an expert sees
// few tokens, computing C^T[N, M] = B^T[N, K] A^T[K, M] lets the large weight
// dimension fill the MMA's fixed-size slot (M = 128 on tcgen05) while the
// tokens take the flexible one (N = any multiple of 16 up to 256). With the
// mini-sglang MoE chapter's sorted layout padded to 16-row blocks (its
// moe_align_block_size with block_m = 16) an expert's tokens are cut into
// near-equal tiles of at most NMAX rows, so decode (1-2 tokens per expert) pays
// for 16 columns instead of a 128-row block (the chapter's first exercise: with
// BLOCK_M = 64 almost all rows are padding).
//
//   gate_up: D0 = W1[e][n0 .. n0+128) x_tok^T, D1 = W1[e][I+n0 ..) x_tok^T,
//            h[pos, n0 + i] = silu(D0[i, pos]) * D1[i, pos]   (x rows gathered in-kernel)
//   down:    D0/D1 = W2[e][h0 .. h0+256) h_tok^T,
//            y_acc[token(pos), h0 + i] += w(pos) * D[i, pos]
//
// The kernels are written in bytes of K: a K step is one 128-byte row segment of
// both operands, 64 bf16 or 128 FP8-e4m3 values, four MMAs of 32 bytes of K each
// (kind::f16 K=16 or kind::f8f6f4 K=32). The FP8 instance (the low-precision GMM
// article's layer: per-token activation scales, per-channel weight scales, fp32
// accumulation) gathers the per-token codes of x, scales each gate_up accumulator by
// its token's and its channel's scale before the SwiGLU, and folds h's per-row scale
// into the route weight and the down channel scale into the combine.
//
// One CTA per SM, persistent. Warps 0-3 epilogue (TMEM lane = weight row),
// warps 4..3+S producers (gate_up: warp 4+s owns ring slot s: lane 0 sends the
// two weight tiles by TMA, the warp gathers the token rows with cp.async; down:
// one thread sends weights and the h rows by TMA), then one MMA warp that also
// owns TMEM. Each k-step issues two M=128 x N tcgen05.mma sharing the token
// tile. Accumulators are double-buffered when NMAX <= 128.
#include "common.cuh"
#include "ptx.cuh"

#include <cuda.h>

namespace moe {

bool make_tmap_bf16_2d_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, int box_rows);
bool make_tmap_u8_2d_k128_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, int box_rows);

namespace {

constexpr int kSwKB = 128;  // bytes of K per step: one 128-byte swizzle row (64 bf16 or 128 e4m3)
constexpr int kSwM = 128;
constexpr int kSwATile = kSwM * kSwKB;  // 16 KB

enum SwapMode { kSwGateUp = 0, kSwDown = 1 };

template <int NMAX>
struct SwapCfg {
  static constexpr int kBBytes = NMAX * kSwKB;
  static constexpr int kStageBytes = 2 * kSwATile + kBBytes;
  static constexpr int kStages = (196608 / kStageBytes) > 6 ? 6 : (196608 / kStageBytes);
  static constexpr int kProdWarps = kStages;
  static constexpr int kMmaWarp = 4 + kProdWarps;
  static constexpr int kThreads = 32 * (kMmaWarp + 1);
  static constexpr int kBufs = NMAX <= 128 ? 2 : 1;
  static constexpr int kD1Off = NMAX <= 128 ? 128 : 256;  // TMEM column offset of D1 within a buffer
  static constexpr int kStagingBytes = 32 * kSwM * 2;      // gate_up epilogue transpose tile [32 tok][128] bf16
  static constexpr int kCtlBytes = 512 + 4 * (MOE_MAX_EXPERTS + 1) + kProdWarps * NMAX * 4 + 3 * NMAX * 4;
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * kStageBytes + kStagingBytes + kCtlBytes;
};

struct SwapArgs {
  const uint8_t* x;            // gate_up: [T, H] bf16 or e4m3 codes (bytes)
  const float* sx;             // FP8 gate_up: per-token scales of x [T]
  const float* sa;             // FP8 down: per-row scales of h [cap]
  const float* sw;             // FP8: per-channel weight scales [E, a_rows_per_expert]
  const int32_t* sorted_ids;   // [cap] (16-row blocks)
  const int32_t* offsets;      // [E + 1] padded segment starts (multiples of 16)
  const float* topk_w;         // down: [num_pairs]
  __nv_bfloat16* h;            // gate_up out: [cap, I]
  float* y_acc;                // down out: [T, H]
  int* err;
  int num_pairs, topk, E, K, I, H;  // K: reduction length in bytes
  int n_wb;                    // weight blocks per expert
  int a_rows_per_expert;       // 2I or H
  int a1_offset;               // row offset of the second weight tile (I for gate_up, 128 for down)
  int wb_stride;               // rows between weight blocks (128 for gate_up, 256 for down)
};

struct SwapTile {
  int e, wb, row0, n;
};

// Token tiles of expert e: its padded length L (multiple of 16) cut into
// ceil(L / NMAX) near-equal tiles whose lengths are multiples of 16.
template <int NMAX>
__device__ __forceinline__ void expert_tiles(int L, int& ntb, int& per) {
  ntb = (L + NMAX - 1) / NMAX;
  per = ntb > 0 ? ((L + ntb - 1) / ntb + 15) / 16 * 16 : 0;
}

template <int NMAX>
__device__ __forceinline__ SwapTile decode_swap(const int* pfx, const SwapArgs& a, int t) {
  // tasks of expert e: n_wb * ntb(e), weight block major, token tile minor
  int lo = 0, hi = a.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pfx[mid] <= t) lo = mid; else hi = mid;
  }
  while (lo + 1 < a.E && pfx[lo + 1] <= t) ++lo;
  SwapTile st;
  st.e = lo;
  const int o0 = __ldg(a.offsets + lo), L = __ldg(a.offsets + lo + 1) - o0;
  int ntb, per;
  expert_tiles<NMAX>(L, ntb, per);
  const int local = t - pfx[lo];
  st.wb = local / ntb;
  const int tb = local - st.wb * ntb;
  st.row0 = o0 + tb * per;
  st.n = min(per, L - tb * per);
  return st;
}

template <int MODE, int NMAX, bool F8>
__global__ void __launch_bounds__(SwapCfg<NMAX>::kThreads, 1)
    moe_swap_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_b,
                    const SwapArgs args) {
  using C = SwapCfg<NMAX>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;  // stage s: [A0 16 KB | A1 16 KB | B NMAX x 128 B]
  __nv_bfloat16* hstage = reinterpret_cast<__nv_bfloat16*>(smem + C::kStages * C::kStageBytes);
  uint8_t* ctl = smem + C::kStages * C::kStageBytes + C::kStagingBytes;
  const uint32_t bar0 = ptx::smem_u32(ctl);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (8 + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (16 + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (18 + b); };
  const uint32_t done_bar = bar0 + 8u * 20;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl + 260);
  int* pfx = reinterpret_cast<int*>(ctl + 512);                                   // [E + 1] task prefix
  int* rowtabs = pfx + (MOE_MAX_EXPERTS + 1);                                     // [kProdWarps][NMAX]
  int* tok_s = rowtabs + C::kProdWarps * NMAX;                                    // [NMAX] epilogue token
  float* w_s = reinterpret_cast<float*>(tok_s + NMAX);                            // [NMAX] epilogue weight
  float* sx_s = w_s + NMAX;                                                       // [NMAX] FP8: token scales

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(full_bar(s), MODE == kSwGateUp ? 32 + 1 : 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), 128);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    ptx::tmem_relinquish();
  } else if (warp == 4) {
    ptx::prefetch_tmap(&map_w);
    if (MODE == kSwDown) ptx::prefetch_tmap(&map_b);
  }
  pdl_wait();  // from here on: reads of what the kernels before this one wrote
  if (warp == 1) {
    // task prefix over experts: pfx[e] = sum_{e' < e} n_wb * ntb(e')
    const int per_lane = (args.E + 31) / 32;
    const int e0 = lane * per_lane;
    int sum = 0;
    for (int j = 0; j < per_lane; ++j) {
      const int e = e0 + j;
      if (e < args.E) {
        int ntb, per;
        expert_tiles<NMAX>(__ldg(args.offsets + e + 1) - __ldg(args.offsets + e), ntb, per);
        sum += ntb * args.n_wb;
      }
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - sum;
    for (int j = 0; j < per_lane; ++j) {
      const int e = e0 + j;
      if (e < args.E) {
        pfx[e] = run;
        int ntb, per;
        expert_tiles<NMAX>(__ldg(args.offsets + e + 1) - __ldg(args.offsets + e), ntb, per);
        run += ntb * args.n_wb;
      }
    }
    if (lane == 31) pfx[args.E] = incl;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int tasks = pfx[args.E];
  const int kblocks = args.K / kSwKB;

  if (warp >= 4 && warp < C::kMmaWarp) {
    // ------------------------------------------------------------ producers
    const int pw = warp - 4;
    if (MODE == kSwGateUp) {
      const int slot = pw;
      int* rowtab = rowtabs + pw * NMAX;  // element offset of each token row of the tile, -1 = pad
      int cached_t = -1, fills = 0;
      SwapTile st{0, 0, 0, 0};
      const uint32_t a_dst = sbase + slot * C::kStageBytes;
      const uint32_t b_dst = a_dst + 2 * kSwATile;
      const int chunk = lane & 7;
      const int rsub = lane >> 3;
      for (int g = slot;; g += C::kStages) {
        const int t_local = g / kblocks;
        const int t = blockIdx.x + t_local * gridDim.x;
        if (t >= tasks) break;
        const int kb = g - t_local * kblocks;
        if (t != cached_t) {
          st = decode_swap<NMAX>(pfx, args, t);
          for (int j = lane; j < NMAX; j += 32) {
            int off = -1;
            if (j < st.n) {
              const int sid = __ldg(args.sorted_ids + st.row0 + j);
              off = (sid < args.num_pairs) ? (sid / args.topk) * args.K : -1;
            }
            rowtab[j] = off;
          }
          cached_t = t;
          __syncwarp();
        }
        const uint32_t use = static_cast<uint32_t>(g / C::kStages);
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(empty_bar(slot), (use & 1u) ^ 1u, abort_flag))) break;
        if (lane == 0) {
          const int wrow = st.e * args.a_rows_per_expert + st.wb * args.wb_stride;
          ptx::mbar_arrive_expect_tx(full_bar(slot), 2 * kSwATile);
          ptx::tma_load_2d(a_dst, &map_w, full_bar(slot), kb * kSwKB / (F8 ? 1 : 2), wrow);
          ptx::tma_load_2d(a_dst + kSwATile, &map_w, full_bar(slot), kb * kSwKB / (F8 ? 1 : 2),
                           wrow + args.a1_offset);
          ++fills;
        }
        const int k0 = kb * kSwKB + chunk * 16;  // bytes
        for (int r = rsub; r < st.n; r += 4) {
          const int off = rowtab[r];
          const uint32_t dst = b_dst + r * 128 + ((chunk ^ (r & 7)) << 4);
          ptx::cp_async_16(dst, off >= 0 ? args.x + off + k0 : args.x, off >= 0 ? 16u : 0u);
        }
        ptx::cp_async_commit();
        ptx::cp_async_wait<0>();
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(full_bar(slot));
      }
      ptx::cp_async_wait<0>();
      if (lane == 0 && fills > 0) ptx::mbar_wait_drain(full_bar(slot), (fills - 1) & 1);
    } else if (pw == 0 && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      bool ok = true;
      for (int t = blockIdx.x; t < tasks && ok; t += gridDim.x) {
        const SwapTile st = decode_swap<NMAX>(pfx, args, t);
        const int wrow = st.e * args.a_rows_per_expert + st.wb * args.wb_stride;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t a_dst = sbase + stage * C::kStageBytes;
          ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * kSwATile + C::kBBytes);
          const int kc = kb * kSwKB / (F8 ? 1 : 2);  // K coordinate in elements
          ptx::tma_load_2d(a_dst, &map_w, full_bar(stage), kc, wrow);
          ptx::tma_load_2d(a_dst + kSwATile, &map_w, full_bar(stage), kc, wrow + args.a1_offset);
          ptx::tma_load_2d(a_dst + 2 * kSwATile, &map_b, full_bar(stage), kc, st.row0);
          ++fills[stage];
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < C::kStages; ++s)
        if (fills[s] > 0) ptx::mbar_wait_drain(full_bar(s), (fills[s] - 1) & 1);
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (ptx::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tasks && ok; t += gridDim.x, ++it) {
        const SwapTile st = decode_swap<NMAX>(pfx, args, t);
        const uint32_t idesc = F8 ? ptx::idesc_e4m3_f32(kSwM, st.n) : ptx::idesc_bf16_f32(kSwM, st.n);
        const int b = C::kBufs == 2 ? (it & 1) : 0;
        const uint32_t tph = C::kBufs == 2 ? ((it >> 1) & 1) : (it & 1);
        if (!ptx::mbar_wait(tempty_bar(b), tph ^ 1u, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t d0 = tmem_base + b * 256, d1 = d0 + C::kD1Off;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t s0 = sbase + stage * C::kStageBytes;
          const uint64_t a0 = ptx::sdesc_sw128(s0), a1 = ptx::sdesc_sw128(s0 + kSwATile);
          const uint64_t bd = ptx::sdesc_sw128(s0 + 2 * kSwATile);
#pragma unroll
          for (int kk = 0; kk < kSwKB / 32; ++kk) {  // 32 bytes of K per MMA
            if constexpr (F8) {
              ptx::mma_f8(d0, a0 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
              ptx::mma_f8(d1, a1 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
            } else {
              ptx::mma_f16(d0, a0 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
              ptx::mma_f16(d1, a1 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
            }
          }
          ptx::mma_commit(empty_bar(stage));
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) ptx::mma_commit(tfull_bar(b));
      }
      ptx::mma_commit(done_bar);
      ptx::mbar_wait_drain(done_bar, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-3, one weight row per thread)
    const int i = warp * 32 + lane;  // row within the 128-row weight tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    int it = 0;
    for (int t = blockIdx.x; t < tasks; t += gridDim.x, ++it) {
      const SwapTile st = decode_swap<NMAX>(pfx, args, t);
      const int b = C::kBufs == 2 ? (it & 1) : 0;
      const uint32_t tph = C::kBufs == 2 ? ((it >> 1) & 1) : (it & 1);
      // per-tile token table (token index, route weight) for the down epilogue; FP8: the
      // route weight times h's row scale (down), the token scales of x (gate_up)
      if (MODE == kSwDown || F8) {
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int j = i; j < st.n; j += 128) {
          const int sid = __ldg(args.sorted_ids + st.row0 + j);
          const bool valid = sid < args.num_pairs;
          if (MODE == kSwDown) {
            tok_s[j] = valid ? sid / args.topk : -1;
            float w = valid ? __ldg(args.topk_w + sid) : 0.f;
            if (F8) w *= valid ? __ldg(args.sa + st.row0 + j) : 0.f;
            w_s[j] = w;
          } else {
            sx_s[j] = valid ? __ldg(args.sx + sid / args.topk) : 0.f;
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
      // FP8: this lane's two channel scales (rows i and a1_offset + i of the weight block)
      float cs0 = 1.f, cs1 = 1.f;
      if (F8) {
        const float* sw = args.sw + static_cast<size_t>(st.e) * args.a_rows_per_expert + st.wb * args.wb_stride;
        cs0 = __ldg(sw + i);
        cs1 = __ldg(sw + args.a1_offset + i);
      }
      // the four warps meet at named barriers in this loop, so they leave it together
      const bool full = ptx::mbar_wait(tfull_bar(b), tph, abort_flag);
      if (ptx::bar_any(1, 128, !full)) break;
      ptx::tc_fence_after();
      const uint32_t d0 = tmem_base + lane_off + b * 256, d1 = d0 + C::kD1Off;
      for (int c = 0; c * 32 < st.n; ++c) {
        uint32_t v0[32], v1[32];
        ptx::tmem_ld32(d0 + c * 32, v0);
        ptx::tmem_ld32(d1 + c * 32, v1);
        ptx::tmem_ld_wait();
        const int jn = min(32, st.n - c * 32);
        if (MODE == kSwGateUp) {
          // h[row0 + c*32 + j, n0 + i] for j < jn, transposed through [32 tok][128] bf16
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float g = __uint_as_float(v0[j]), u = __uint_as_float(v1[j]);
            if (F8) {
              // g = sx[token] * sw[e, n] * acc_g, u = sx[token] * sw[e, I + n] * acc_u
              const float rs = sx_s[c * 32 + j];
              g = rs * cs0 * g;
              u = rs * cs1 * u;
            }
            hstage[j * kSwM + i] = __float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * u);
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
          // 16 lanes store one token's 256 bytes: a warp covers 2 tokens per instruction
          const int n0 = st.wb * kSwM;
          for (int j = warp * 2 + (lane >> 4); j < jn; j += 8) {
            const uint4 val = reinterpret_cast<const uint4*>(hstage + j * kSwM)[lane & 15];
            reinterpret_cast<uint4*>(args.h + static_cast<size_t>(st.row0 + c * 32 + j) * args.I + n0)[lane & 15] =
                val;
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
        } else {
          // y_acc[token, h0 + i] += w * D: for each token a warp adds 32 consecutive floats
          const int h0 = st.wb * 2 * kSwM;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tok = tok_s[c * 32 + j];
            if (j < jn && tok >= 0) {
              const float w = w_s[c * 32 + j];
              float* yrow = args.y_acc + static_cast<size_t>(tok) * args.H + h0;
              if (F8) {  // w * sh[row] (folded in w_s) * sw[e, channel] * acc
                atomicAdd(yrow + i, (w * cs0) * __uint_as_float(v0[j]));
                atomicAdd(yrow + kSwM + i, (w * cs1) * __uint_as_float(v1[j]));
              } else {
                atomicAdd(yrow + i, w * __uint_as_float(v0[j]));
                atomicAdd(yrow + kSwM + i, w * __uint_as_float(v1[j]));
              }
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty_bar(b));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == C::kMmaWarp) ptx::tmem_dealloc(tmem_base, 512);
  if (tid == 0 && *abort_flag) report_error(args.err, MOE_DEVERR_TIMEOUT);
}

template <int MODE, int NMAX, bool F8>
moe_status_t launch_swap_impl(const CUtensorMap& mw, const CUtensorMap& mb, const SwapArgs& a, cudaStream_t s) {
  using C = SwapCfg<NMAX>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(moe_swap_kernel<MODE, NMAX, F8>), static_cast<int>(C::kSmem)))
    return MOE_ERR_CUDA;
  return launch_pdl(moe_swap_kernel<MODE, NMAX, F8>, dim3(num_sms()), dim3(C::kThreads), C::kSmem, s, mw, mb, a);
}

}  // namespace

// nmax: token tile cap (32 for decode-sized problems, 256 otherwise).
moe_status_t launch_swap_gate_up(const __nv_bfloat16* x, const __nv_bfloat16* w1, const int32_t* sorted_ids,
                                 const int32_t* offsets, __nv_bfloat16* h, int* err, int num_pairs, int topk, int H,
                                 int I, int E, int nmax, cudaStream_t s) {
  CUtensorMap mw;
  if (!make_tmap_bf16_2d_rows(&mw, w1, static_cast<uint64_t>(E) * 2 * I, H, kSwM)) return MOE_ERR_CUDA;
  SwapArgs a{};
  a.x = reinterpret_cast<const uint8_t*>(x); a.sorted_ids = sorted_ids; a.offsets = offsets; a.h = h; a.err = err;
  a.num_pairs = num_pairs; a.topk = topk; a.E = E; a.K = 2 * H; a.I = I; a.H = H;
  a.n_wb = I / kSwM; a.a_rows_per_expert = 2 * I; a.a1_offset = I; a.wb_stride = kSwM;
  if (nmax <= 32) return launch_swap_impl<kSwGateUp, 32, false>(mw, mw, a, s);
  return launch_swap_impl<kSwGateUp, 256, false>(mw, mw, a, s);
}

moe_status_t launch_swap_down(const __nv_bfloat16* h, const __nv_bfloat16* w2, const int32_t* sorted_ids,
                              const int32_t* offsets, const float* topk_w, float* y_acc, int* err, int num_pairs,
                              int topk, int cap, int H, int I, int E, int nmax, cudaStream_t s) {
  CUtensorMap mw, mb;
  const int box = nmax <= 32 ? 32 : 256;
  if (!make_tmap_bf16_2d_rows(&mw, w2, static_cast<uint64_t>(E) * H, I, kSwM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d_rows(&mb, h, static_cast<uint64_t>(cap), I, box)) return MOE_ERR_CUDA;
  SwapArgs a{};
  a.sorted_ids = sorted_ids; a.offsets = offsets; a.topk_w = topk_w; a.y_acc = y_acc; a.err = err;
  a.num_pairs = num_pairs; a.topk = topk; a.E = E; a.K = 2 * I; a.I = I; a.H = H;
  a.n_wb = H / (2 * kSwM); a.a_rows_per_expert = H; a.a1_offset = kSwM; a.wb_stride = 2 * kSwM;
  if (nmax <= 32) return launch_swap_impl<kSwDown, 32, false>(mw, mb, a, s);
  return launch_swap_impl<kSwDown, 256, false>(mw, mb, a, s);
}

// FP8-e4m3 operands (decode-sized problems: token tiles of <= 32). qx: per-token codes
// of x [T, H] with scales sx [T]; w1: codes [E, 2I, H] with per-channel scales sw1 [E, 2I].
moe_status_t launch_swap_gate_up_fp8(const uint8_t* qx, const float* sx, const uint8_t* w1, const float* sw1,
                                     const int32_t* sorted_ids, const int32_t* offsets, __nv_bfloat16* h, int* err,
                                     int num_pairs, int topk, int H, int I, int E, cudaStream_t s) {
  CUtensorMap mw;
  if (!make_tmap_u8_2d_k128_rows(&mw, w1, static_cast<uint64_t>(E) * 2 * I, H, kSwM)) return MOE_ERR_CUDA;
  SwapArgs a{};
  a.x = qx; a.sx = sx; a.sw = sw1; a.sorted_ids = sorted_ids; a.offsets = offsets; a.h = h; a.err = err;
  a.num_pairs = num_pairs; a.topk = topk; a.E = E; a.K = H; a.I = I; a.H = H;
  a.n_wb = I / kSwM; a.a_rows_per_expert = 2 * I; a.a1_offset = I; a.wb_stride = kSwM;
  return launch_swap_impl<kSwGateUp, 32, true>(mw, mw, a, s);
}

// qh: per-row codes of h [cap, I] with scales sh [cap]; w2: codes [E, H, I] with sw2 [E, H].
moe_status_t launch_swap_down_fp8(const uint8_t* qh, const float* sh, const uint8_t* w2, const float* sw2,
                                  const int32_t* sorted_ids, const int32_t* offsets, const float* topk_w,
                                  float* y_acc, int* err, int num_pairs, int topk, int cap, int H, int I, int E,
                                  cudaStream_t s) {
  CUtensorMap mw, mb;
  if (!make_tmap_u8_2d_k128_rows(&mw, w2, static_cast<uint64_t>(E) * H, I, kSwM)) return MOE_ERR_CUDA;
  if (!make_tmap_u8_2d_k128_rows(&mb, qh, static_cast<uint64_t>(cap), I, 32)) return MOE_ERR_CUDA;
  SwapArgs a{};
  a.sa = sh; a.sw = sw2; a.sorted_ids = sorted_ids; a.offsets = offsets; a.topk_w = topk_w; a.y_acc = y_acc;
  a.err = err; a.num_pairs = num_pairs; a.topk = topk; a.E = E; a.K = I; a.I = I; a.H = H;
  a.n_wb = H / (2 * kSwM); a.a_rows_per_expert = H; a.a1_offset = kSwM; a.wb_stride = 2 * kSwM;
  return launch_swap_impl<kSwDown, 32, true>(mw, mb, a, s);
}

}  // namespace moe
