// down grouped GEMM of the MoE layer over the expert-sorted, BLOCK_M-padded pair
// layout, on tcgen05 tensor cores with TMEM accumulators, and the 2D tensor maps
// (TMA descriptors) of the grouped GEMM kernels.
//
// Follows the mini-sglang MoE chapter ("fused MoE", fused_moe_kernel and
// FusedMoeBackend.forward, second launch): every 128-row block of the sorted
// layout belongs to one expert (expert_ids), its rows are the pairs
// sorted_token_ids[...], and C[row] = h[row] @ W2[e]^T is scaled by the route
// weight of the row's pair and summed into the pair's token row of the fp32
// accumulator. h is contiguous per expert (the gate_up kernels write it in
// sorted order), so both operands arrive by TMA.
//
// Kernel shape (one persistent CTA per SM, 320 threads):
//   warps 0-(P-1)  epilogue: TMEM -> registers -> shared staging -> fp32 reductions
//              (red.global.add, L2 evict-last)
//              (TMEM lane quarter = warp % 4). The bf16 instance has P = 4 warps;
//              the FP8 instance P = 8 (column half = warp / 4: two warps drain
//              each accumulator row), so that the combine of a tile stays shorter
//              than the main loop of the next, which FP8 operands halve. (Eight
//              warps made the bf16 instance 4 % slower.)
//   warp P     one thread sends A and B of every K step by TMA through the
//              4-slot ring
//   warp P+1   TMEM allocation and the single MMA-issuing thread
// The kernel is written in bytes of K: a K step is one 128-byte swizzle row of
// both operands (64 bf16 or 128 FP8-e4m3 values), four MMAs of 32 bytes of K.
// The FP8 instance (the low-precision GMM article's layer: per-token
// activation scales, per-channel weight scales, sections 2.3 and 4.3) reads h
// quantised per row and multiplies each accumulator by its row's scale and its
// column's weight scale in the epilogue, together with the route weight.
// The 128 x 256 fp32 accumulator lives in TMEM, double-buffered (512 columns)
// so that the combine of one tile overlaps the main loop of the next.
// Tiles (m-block, n-block) are taken round-robin with the n-block fastest, so
// the CTAs working at one time share each expert's weight tiles through L2.
#include "common.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

namespace moe {

constexpr int kBM = 128;          // rows per tile (= align block_m)
constexpr int kBN = 256;          // accumulator columns per tile
constexpr int kBK = 64;           // K per stage (128 bytes of bf16: one swizzle row)
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBytes = kBN * kBK * 2;   // 32 KB
template <bool F8> constexpr int epi_threads() { return F8 ? 256 : 128; }
constexpr int kProdThreads = 32;
template <bool F8> constexpr int gemm_threads() { return epi_threads<F8>() + kProdThreads + 32; }
constexpr int kTmemCols = 2 * kBN;
// Staging tile of one epilogue warp: 32 rows x 32 floats, the 16-byte slot q of
// row r stored at slot q ^ (r & 7) (conflict-free row-wise writes and 8-lane
// row reads without padding).
constexpr size_t kEpiStageBytes = (epi_threads<true>() / 32) * 32 * 32 * 4;  // sized for the larger instance
constexpr size_t kGemmSmem = 1024 + kStages * (kABytes + kBBytes) + 256 + kEpiStageBytes;

struct GemmArgs {
  const int32_t* sorted_ids;      // [cap] pair index or sentinel num_pairs
  const int32_t* expert_ids;      // [cap / 128]
  const int32_t* ntpp;            // [1] padded rows in use
  const float* topk_w;            // [num_pairs] route weights
  const float* sa;                // FP8: per-row scales of the A operand [cap]
  const float* sw;                // FP8: per-channel weight scales [E, H]
  float* y_acc;                   // [T, H] fp32 accumulator
  int* err;
  int num_pairs, topk;
  int K;                          // reduction length (I), in elements
  int H;
  int n_tiles;                    // n-blocks per m-block
  int b_rows_per_expert;          // rows of the 2D weight view per expert (H)
};

template <bool F8>
__global__ void __launch_bounds__(gemm_threads<F8>(), 1)
    moe_down_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const GemmArgs args) {
  constexpr int kElemsPerStep = F8 ? 2 * kBK : kBK;  // K elements per 128-byte step
  constexpr int kEpiThreads = epi_threads<F8>();
  constexpr int kMmaWarp = (kEpiThreads + kProdThreads) / 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sA = raw_addr + pad;                       // kStages x 16 KB
  const uint32_t sB = sA + kStages * kABytes;               // kStages x 32 KB
  uint8_t* ctl = smem + kStages * (kABytes + kBBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ctl);
  // bars: full[kStages], empty[kStages], tfull[2], tempty[2], done
  const uint32_t bar_base = ptx::smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * (2 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * (2 * kStages + 2 + b); };
  const uint32_t done_bar = bar_base + 8u * (2 * kStages + 4);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl + 132);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), kEpiThreads);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (tid == kEpiThreads) {
    ptx::prefetch_tmap(&map_b);
    ptx::prefetch_tmap(&map_a);
  }
  pdl_wait();  // from here on: reads of what the kernels before this one wrote
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int m_tiles = __ldg(args.ntpp) / kBM;
  const int tiles = m_tiles * args.n_tiles;
  const int kblocks = args.K / kElemsPerStep;

  if (warp == kEpiThreads / 32) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int mt = t / args.n_tiles;
        const int nt = t - mt * args.n_tiles;
        const int e = __ldg(args.expert_ids + mt);
        const int b_row0 = e * args.b_rows_per_expert + nt * kBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t a_dst = sA + stage * kABytes;
          const uint32_t b_dst = sB + stage * kBBytes;
          ptx::mbar_arrive_expect_tx(full_bar(stage), kBBytes + kABytes);
          ptx::tma_load_2d(b_dst, &map_b, full_bar(stage), kb * kElemsPerStep, b_row0);
          ptx::tma_load_2d(b_dst + kBBytes / 2, &map_b, full_bar(stage), kb * kElemsPerStep, b_row0 + kBM);
          ptx::tma_load_2d(a_dst, &map_a, full_bar(stage), kb * kElemsPerStep, mt * kBM);
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
#pragma unroll
      for (int st = 0; st < kStages; ++st) {
        const int fills = issued / kStages + (st < issued % kStages ? 1 : 0);
        if (fills > 0) ptx::mbar_wait_drain(full_bar(st), (fills - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (ptx::elect_one()) {
      constexpr uint32_t idesc = F8 ? ptx::idesc_e4m3_f32(kBM, kBN) : ptx::idesc_bf16_f32(kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++it) {
        const int b = it & 1;
        const uint32_t tphase = (it >> 1) & 1;
        if (!ptx::mbar_wait(tempty_bar(b), tphase ^ 1u, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t adesc = ptx::sdesc_sw128(sA + stage * kABytes);
          const uint64_t bdesc = ptx::sdesc_sw128(sB + stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of K per MMA
            if constexpr (F8) ptx::mma_f8(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
            else ptx::mma_f16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
          }
          ptx::mma_commit(empty_bar(stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) ptx::mma_commit(tfull_bar(b));
      }
      // all issued MMAs complete before TMEM is released
      ptx::mma_commit(done_bar);
      ptx::mbar_wait_drain(done_bar, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Each warp drains its 32 accumulator rows 32 columns at a time through a
    // shared staging tile, so that the fp32 atomics of one instruction cover
    // whole 128-byte row segments of 4 rows instead of 32 scattered 16-byte
    // pieces.
    float4* stg = reinterpret_cast<float4*>(ctl + 256) + warp * 32 * 8;
    constexpr int kParts = kEpiThreads / 128;  // warps per TMEM lane quarter
    const int quarter = warp & 3;
    const int chalf = warp >> 2;     // accumulator columns [kBN / kParts * chalf, ...) of this warp
    const int r = quarter * 32 + lane;  // accumulator row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // The accumulator rows are reduced into at L2 while the weights stream past:
    // evict-last keeps them resident.
    const uint64_t acc_pol = ptx::l2_policy_evict_last();
    int it = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
      const int b = it & 1;
      const uint32_t tphase = (it >> 1) & 1;
      const int mt = t / args.n_tiles;
      const int nt = t - mt * args.n_tiles;
      const int pos = mt * kBM + r;
      // the row's pair, token and weights are loaded before waiting for the accumulator
      const int sid = __ldg(args.sorted_ids + pos);
      const bool valid = sid < args.num_pairs;
      float w = valid ? __ldg(args.topk_w + sid) : 0.f;
      if constexpr (F8) w *= valid ? __ldg(args.sa + pos) : 0.f;  // and the row's quantisation scale
      const int tok = valid ? sid / args.topk : -1;
      const int e_of_tile = F8 ? __ldg(args.expert_ids + mt) : 0;
      // the warp leaves as one (warp-wide TMEM loads and shuffles follow)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(tfull_bar(b), tphase, abort_flag))) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + lane_off + b * kBN;
      // Two forms of the combine loop, each the faster one measured for its operand type: the
      // FP8 instance hoists the token rows and loads the channel scales a chunk ahead (its
      // main loop is half as long, so the combine's chain bounds it); the bf16 instance keeps
      // the plain loop, which was 4 % faster for it.
      if constexpr (F8) {
        // The TMEM load of the next 32 columns is issued as soon as the current
        // one has landed, so that it overlaps this chunk's scaling, staging and
        // atomics (FP8 tiles have half the main loop to hide the combine behind).
        constexpr int kCh = kBN / 32 / kParts;  // 32-column chunks per warp
        const int c0 = chalf * kCh;
        // the token row each lane adds into, for its 8 (row, 16-byte) slots of a chunk
        int trow[8];
  #pragma unroll
        for (int i = 0; i < 8; ++i) trow[i] = __shfl_sync(0xffffffffu, tok, i * 4 + (lane >> 3));
        // FP8: the chunk's 32 channel scales, loaded one chunk ahead
        const float4* swt = F8 ? reinterpret_cast<const float4*>(args.sw + static_cast<size_t>(e_of_tile) * args.H +
                                                                  nt * kBN + c0 * 32)
                               : nullptr;
        float4 cs[2][8];
        if constexpr (F8) {
  #pragma unroll
          for (int q = 0; q < 8; ++q) cs[0][q] = __ldg(swt + q);
        }
        uint32_t d[2][32];
        ptx::tmem_ld32(tbase + c0 * 32, d[0]);
  #pragma unroll
        for (int ci = 0; ci < kCh; ++ci) {
          const int c = c0 + ci;
          if constexpr (F8) {
            if (ci + 1 < kCh) {
  #pragma unroll
              for (int q = 0; q < 8; ++q) cs[(ci + 1) & 1][q] = __ldg(swt + 8 * (ci + 1) + q);
            }
          }
          ptx::tmem_ld_wait();
          if (ci + 1 < kCh) ptx::tmem_ld32(tbase + (c + 1) * 32, d[(ci + 1) & 1]);
          const uint32_t* dc = d[ci & 1];
          const float4* csc = cs[ci & 1];
          float4 srow[8];
  #pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 k = F8 ? make_float4(w * csc[q].x, w * csc[q].y, w * csc[q].z, w * csc[q].w)
                                : make_float4(w, w, w, w);
            srow[q] = make_float4(k.x * __uint_as_float(dc[4 * q]), k.y * __uint_as_float(dc[4 * q + 1]),
                                  k.z * __uint_as_float(dc[4 * q + 2]), k.w * __uint_as_float(dc[4 * q + 3]));
          }
  #pragma unroll
          for (int q = 0; q < 8; ++q) stg[lane * 8 + (q ^ (lane & 7))] = srow[q];
          __syncwarp();
          // 8 lanes add one row's 32 floats (128 contiguous bytes) into its token row
  #pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = i * 4 + (lane >> 3);
            const int q = lane & 7;
            const float4 v = stg[rl * 8 + (q ^ (rl & 7))];
            if (trow[i] >= 0)
              ptx::red_add_f32x4(args.y_acc + static_cast<size_t>(trow[i]) * args.H + nt * kBN + c * 32 + 4 * q, v,
                                 acc_pol);
          }
          __syncwarp();
        }
      } else {
        // The TMEM load of the next 32 columns is issued as soon as the current
        // one has landed, so that it overlaps this chunk's scaling, staging and
        // atomics; the token row is shuffled per row (bf16 tiles have the longer
        // main loop, which hides this combine).
        constexpr int kCh = kBN / 32 / kParts;  // 32-column chunks per warp
        const int c0 = chalf * kCh;
        uint32_t d[2][32];
        ptx::tmem_ld32(tbase + c0 * 32, d[0]);
  #pragma unroll
        for (int ci = 0; ci < kCh; ++ci) {
          const int c = c0 + ci;
          ptx::tmem_ld_wait();
          if (ci + 1 < kCh) ptx::tmem_ld32(tbase + (c + 1) * 32, d[(ci + 1) & 1]);
          const uint32_t* dc = d[ci & 1];
          float4 srow[8];
  #pragma unroll
          for (int q = 0; q < 8; ++q)
            srow[q] = make_float4(w * __uint_as_float(dc[4 * q]), w * __uint_as_float(dc[4 * q + 1]),
                                  w * __uint_as_float(dc[4 * q + 2]), w * __uint_as_float(dc[4 * q + 3]));
  #pragma unroll
          for (int q = 0; q < 8; ++q) stg[lane * 8 + (q ^ (lane & 7))] = srow[q];
          __syncwarp();
          // 8 lanes add one row's 32 floats (128 contiguous bytes) into its token row
  #pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = i * 4 + (lane >> 3);
            const int q = lane & 7;
            const int trow = __shfl_sync(0xffffffffu, tok, rl);
            const float4 v = stg[rl * 8 + (q ^ (rl & 7))];
            if (trow >= 0)
              ptx::red_add_f32x4(args.y_acc + static_cast<size_t>(trow) * args.H + nt * kBN + c * 32 + 4 * q, v,
                                 acc_pol);
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty_bar(b));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem_base, kTmemCols);
  if (tid == 0 && *abort_flag) report_error(args.err, MOE_DEVERR_TIMEOUT);
}

// ----------------------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// 2D bf16 tensor map over a row-major [rows, cols] matrix, box = 64 cols x 128 rows, 128B swizzle.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
  auto encode = get_encode_fn();
  if (!encode) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBM)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Same with a chosen box height (rows per load, <= 256).
bool make_tmap_bf16_2d_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, int box_rows) {
  auto encode = get_encode_fn();
  if (!encode || box_rows < 1 || box_rows > 256) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Same with a box of 32 columns (64 bytes) x 128 rows and 64B swizzle.
bool make_tmap_bf16_2d_k32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
  auto encode = get_encode_fn();
  if (!encode) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kBM)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2D 8-bit tensor map, box = 64 columns (bytes) x 128 rows, 64B swizzle.
bool make_tmap_u8_2d_k64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
  auto encode = get_encode_fn();
  if (!encode) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2D 8-bit tensor map over a row-major [rows, cols] byte matrix, box = 128 x 128,
// 128B swizzle (tcgen05 operand) or none (staging read back by threads).
bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, bool swizzle128) {
  auto encode = get_encode_fn();
  if (!encode) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE,
                            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <bool F8>
moe_status_t launch_down(const CUtensorMap& map_a, const CUtensorMap& map_b, const GemmArgs& a, cudaStream_t s) {
  if (!ensure_smem_attr(reinterpret_cast<const void*>(moe_down_kernel<F8>), static_cast<int>(kGemmSmem)))
    return MOE_ERR_CUDA;
  return launch_pdl(moe_down_kernel<F8>, dim3(num_sms()), dim3(gemm_threads<F8>()), kGemmSmem, s, map_a, map_b, a);
}

}  // namespace

moe_status_t launch_gemm_down(const __nv_bfloat16* h, const __nv_bfloat16* w2, const int32_t* sorted_ids,
                              const int32_t* expert_ids, const int32_t* ntpp, const float* topk_w, float* y_acc,
                              int* err, int num_pairs, int topk, int cap, int H, int I, int E, cudaStream_t s) {
  CUtensorMap map_a, map_b;
  if (!make_tmap_bf16_2d(&map_a, h, static_cast<uint64_t>(cap), I)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&map_b, w2, static_cast<uint64_t>(E) * H, I)) return MOE_ERR_CUDA;
  GemmArgs a{};
  a.sorted_ids = sorted_ids; a.expert_ids = expert_ids; a.ntpp = ntpp; a.topk_w = topk_w; a.y_acc = y_acc;
  a.err = err; a.num_pairs = num_pairs; a.topk = topk; a.K = I; a.H = H;
  a.n_tiles = H / kBN; a.b_rows_per_expert = H;
  return launch_down<false>(map_a, map_b, a, s);
}

moe_status_t launch_gemm_down_fp8(const uint8_t* qh, const float* sh, const uint8_t* w2, const float* sw2,
                                  const int32_t* sorted_ids, const int32_t* expert_ids, const int32_t* ntpp,
                                  const float* topk_w, float* y_acc, int* err, int num_pairs, int topk, int cap,
                                  int H, int I, int E, cudaStream_t s) {
  if (I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  CUtensorMap map_a, map_b;
  if (!make_tmap_u8_2d(&map_a, qh, static_cast<uint64_t>(cap), I, true)) return MOE_ERR_CUDA;
  if (!make_tmap_u8_2d(&map_b, w2, static_cast<uint64_t>(E) * H, I, true)) return MOE_ERR_CUDA;
  GemmArgs a{};
  a.sorted_ids = sorted_ids; a.expert_ids = expert_ids; a.ntpp = ntpp; a.topk_w = topk_w; a.y_acc = y_acc;
  a.sa = sh; a.sw = sw2;
  a.err = err; a.num_pairs = num_pairs; a.topk = topk; a.K = I; a.H = H;
  a.n_tiles = H / kBN; a.b_rows_per_expert = H;
  return launch_down<true>(map_a, map_b, a, s);
}

}  // namespace moe
