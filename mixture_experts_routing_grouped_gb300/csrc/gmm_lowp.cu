// gmm_lowp: low-precision grouped GEMM with the scales fused into the epilogue.
//
// Follows the low-precision GMM article (pwwt.cn): section 2.1
// Y_e = X[S_e] W_e^T over the expert-sorted row ranges S_e = [off[e], off[e]+size[e]),
// section 3.1's interface and per-token / per-channel scales applied in-kernel,
// section 2.3's fp32 accumulation, section 3.3's dynamic work queue (every expert
// cut into 128-row tasks, persistent blocks claim tasks from one atomic counter)
// and section 3.4's [E, N, K] weight layout with K contiguous.
//
//   out[m, n] = scales_x[m] * scales_w[e, n] * sum_k q_x[m, k] * q_w[e, n, k]
//
// FP8-e4m3 runs natively on tcgen05 (kind::f8f6f4, fp32 accumulation in TMEM).
// tcgen05 has no integer MMA on sm_103a, so INT8 tiles are brought in by TMA
// unconverted and widened in shared memory to fp16 (exact for |q| <= 128) by
// four converter warps; the MMA is then kind::f16 with fp32 accumulation.
//
// Kernel shape (one persistent CTA per SM): warps 0-3 epilogue, warp 4 task
// claimer + TMA producer, warp 5 TMA-owner of TMEM + MMA issuer, warps 6-9
// INT8 converters. Tile 128 rows x 128 columns x 128 K; a task is (expert,
// 128-row block, 128-column block), ordered expert, column block, row block so
// that CTAs running together share each weight tile in L2. Rows of a block past
// the expert's end are computed on whatever TMA brought (the next expert's rows
// or zero fill) and never stored.
#include "common.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <cuda_fp16.h>

namespace moe {

bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, bool swizzle128);

namespace {

constexpr int kLBM = 128, kLBN = 128, kLBK = 128;      // K in elements (= bytes for 8-bit codes)
constexpr int kTile8 = kLBM * kLBK;                     // 16 KB: one 8-bit operand tile
constexpr int kF8Stages = 6;                            // fp8: 6 x (A 16 KB + B 16 KB)
constexpr int kI8Stages = 2;                            // int8: 2 x 32 KB staging + 2 x 64 KB fp16 operands
constexpr int kTile16 = kLBM * kLBK * 2;                // 32 KB: one fp16 operand tile (2 column blocks)
constexpr int kQ = 4;                                   // task queue slots
constexpr int kLThreads = 320;
constexpr int kLTmemCols = 2 * kLBN;
constexpr size_t kLSmem = 1024 + 192 * 1024 + 512;

struct LowpArgs {
  const float* sx;
  const float* sw;
  const int32_t* offsets;
  const int32_t* sizes;
  const int32_t* mt_prefix;  // [E+1] row blocks before each expert
  int* counter;              // task counter (zeroed by the prep kernel)
  const int* num_tasks;
  void* out;
  int* err;
  int M, K, N, E, out_f32;
};

struct Task {
  int e, row0, rows, nt;
};

// Task t -> (expert, row block, column block). Tasks of one expert are laid out
// column block by column block, row blocks fastest.
__device__ __forceinline__ Task decode_task(const LowpArgs& a, int n_tiles, int t) {
  const int g_tile_task = t;  // tasks before expert e = prefix[e] * n_tiles
  int lo = 0, hi = a.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a.mt_prefix + mid) * n_tiles <= g_tile_task) lo = mid; else hi = mid;
  }
  while (lo + 1 < a.E && __ldg(a.mt_prefix + lo + 1) * n_tiles <= g_tile_task) ++lo;
  Task k;
  k.e = lo;
  const int mcount = __ldg(a.mt_prefix + lo + 1) - __ldg(a.mt_prefix + lo);
  const int local = t - __ldg(a.mt_prefix + lo) * n_tiles;
  k.nt = local / mcount;
  const int mt = local - k.nt * mcount;
  const int off = __ldg(a.offsets + lo);
  const int size = __ldg(a.sizes + lo);
  k.row0 = off + mt * kLBM;
  k.rows = min(kLBM, off + size - k.row0);
  return k;
}

// Validates the group metadata, counts 128-row blocks per expert and zeroes the task counter.
__global__ void __launch_bounds__(1024) lowp_prep_kernel(const int32_t* __restrict__ offsets,
                                                         const int32_t* __restrict__ sizes, int E, int M,
                                                         int n_tiles, int32_t* __restrict__ mt_prefix,
                                                         int* __restrict__ counter, int* __restrict__ num_tasks,
                                                         int* __restrict__ err) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int blocks = 0;
  if (tid < E) {
    const int o0 = offsets[tid], o1 = offsets[tid + 1], s = sizes[tid];
    const bool ok = s >= 0 && o0 >= 0 && o1 <= M && o1 - o0 == s;
    if (!ok) report_error(err, MOE_DEVERR_GROUP_META);
    else blocks = (s + kLBM - 1) / kLBM;
  }
  if (tid == 0 && (offsets[0] != 0 || offsets[E] != M)) report_error(err, MOE_DEVERR_GROUP_META);
  int incl = blocks;
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
  const int excl = incl - blocks + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (tid < E) mt_prefix[tid] = excl;
  if (tid == E - 1) {
    mt_prefix[E] = excl + blocks;
    *num_tasks = (excl + blocks) * n_tiles;
  }
  if (tid == 0) *counter = 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// int8 x4 (one 32-bit word) -> 4 fp16 values, exactly: fp16(0x6400 | (q + 128)) = 1024 + q + 128.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

template <bool I8>
__global__ void __launch_bounds__(kLThreads, 1)
    gmm_lowp_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                    const LowpArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  constexpr int kStages = I8 ? kI8Stages : kF8Stages;
  // fp8: stage s = [A 16 KB | B 16 KB] at s*32 KB.
  // int8: staging s = [A 16 KB | B 16 KB] at s*32 KB (no swizzle); fp16 operands
  //       o = [A 32 KB | B 32 KB] at 64 KB + o*64 KB, each tile = 2 column blocks of
  //       [128 rows][128 B] with the 128B swizzle.
  uint8_t* ctl = smem + 192 * 1024;
  const uint32_t bar0 = ptx::smem_u32(ctl);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };                 // staging / stage landed
  auto empty_bar = [&](int s) { return bar0 + 8u * (8 + s); };          // staging / stage free
  auto ofull_bar = [&](int s) { return bar0 + 8u * (16 + s); };         // int8: fp16 operand ready
  auto oempty_bar = [&](int s) { return bar0 + 8u * (20 + s); };        // int8: fp16 operand free
  auto tfull_bar = [&](int b) { return bar0 + 8u * (24 + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (26 + b); };
  auto qfull_bar = [&](int q) { return bar0 + 8u * (28 + q); };
  auto qempty_bar = [&](int q) { return bar0 + 8u * (32 + q); };
  const uint32_t done_bar = bar0 + 8u * 36;
  volatile int* tq = reinterpret_cast<volatile int*>(ctl + 304);       // [kQ] claimed task ids
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + 320);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl + 324);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = args.N / kLBN;
  const int kblocks = args.K / kLBK;
  const int num_tasks = __ldg(args.num_tasks);
  constexpr int kConsumers = 1 + 128 + (I8 ? 128 : 0);

  if (tid == 0) {
    for (int s = 0; s < 8; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), I8 ? 128 : 1);
    }
    for (int s = 0; s < 4; ++s) {
      ptx::mbar_init(ofull_bar(s), 128);
      ptx::mbar_init(oempty_bar(s), 1);
      ptx::mbar_init(qfull_bar(s), 1);
      ptx::mbar_init(qempty_bar(s), kConsumers);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), 128);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), kLTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Task queue consumer: returns the next task id (>= num_tasks means done) or -1 on abort.
  auto next_task = [&](int it) -> int {
    const int q = it % kQ;
    if (!ptx::mbar_wait(qfull_bar(q), (static_cast<uint32_t>(it / kQ) & 1u), abort_flag)) return -1;
    const int t = tq[q];
    ptx::mbar_arrive(qempty_bar(q));
    return t;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ task claimer + TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int it = 0;; ++it) {
        const int q = it % kQ;
        if (!ptx::mbar_wait(qempty_bar(q), (static_cast<uint32_t>(it / kQ) & 1u) ^ 1u, abort_flag)) break;
        const int t = atomicAdd(args.counter, 1);
        tq[q] = t;
        ptx::mbar_arrive(qfull_bar(q));
        if (t >= num_tasks) break;
        const Task k = decode_task(args, n_tiles, t);
        const int wrow = k.e * args.N + k.nt * kLBN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t dst = sbase + stage * 2 * kTile8;
          ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * kTile8);
          ptx::tma_load_2d(dst, &map_x, full_bar(stage), kb * kLBK, k.row0);
          ptx::tma_load_2d(dst + kTile8, &map_w, full_bar(stage), kb * kLBK, wrow);
          ++fills[stage];
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      for (int s = 0; s < kStages; ++s)
        if (fills[s] > 0) ptx::mbar_wait_drain(full_bar(s), (fills[s] - 1) & 1);
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------------------------------------ int8 -> fp16 converters
    if constexpr (I8) {
      const int c = tid - 192;  // 0..127
      int stage = 0, ostage = 0;
      uint32_t phase = 0, ophase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int t = next_task(it);
        if (t < 0 || t >= num_tasks) break;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          if (!ptx::mbar_wait(oempty_bar(ostage), ophase ^ 1u, abort_flag)) { ok = false; break; }
          const uint8_t* src = smem + stage * 2 * kTile8;
          const uint32_t dst = sbase + 64 * 1024 + ostage * 2 * kTile16;
          // 2 tiles x 128 rows x 8 chunks of 16 bytes; thread c handles chunk (c & 7) of 8 rows per tile
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            const int tile = i >> 3;
            const int r = (c >> 3) + 16 * (i & 7);
            const int ch = c & 7;  // 16 int8 = k in [ch*16, ch*16+16)
            const uint4 v = *reinterpret_cast<const uint4*>(src + tile * kTile8 + r * 128 + ch * 16);
            uint32_t h[8];
            i8x4_to_f16x4(v.x, h[0], h[1]);
            i8x4_to_f16x4(v.y, h[2], h[3]);
            i8x4_to_f16x4(v.z, h[4], h[5]);
            i8x4_to_f16x4(v.w, h[6], h[7]);
            // fp16 k index ch*16 .. +16 -> column block cb = ch / 4, 16-byte chunks j0, j0+1 in the 128-byte row
            const int cb = ch >> 2;
            const int j0 = (ch & 3) * 2;
            const uint32_t rowbase = dst + tile * kTile16 + cb * kTile8 + r * 128;
            const uint32_t d0 = rowbase + (((j0) ^ (r & 7)) << 4);
            const uint32_t d1 = rowbase + (((j0 + 1) ^ (r & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d0), "r"(h[0]), "r"(h[1]), "r"(h[2]),
                         "r"(h[3]) : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d1), "r"(h[4]), "r"(h[5]), "r"(h[6]),
                         "r"(h[7]) : "memory");
          }
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive(ofull_bar(ostage));
          ptx::mbar_arrive(empty_bar(stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
          if (++ostage == 2) { ostage = 0; ophase ^= 1u; }
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (ptx::elect_one()) {
      const uint32_t idesc = I8 ? (ptx::idesc_bf16_f32(kLBM, kLBN) & ~((7u << 7) | (7u << 10)))  // fp16 A/B
                                : ptx::idesc_e4m3_f32(kLBM, kLBN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int t = next_task(it);
        if (t < 0 || t >= num_tasks) break;
        const int b = it & 1;
        if (!ptx::mbar_wait(tempty_bar(b), ((it >> 1) & 1) ^ 1u, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kLBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if constexpr (I8) {
            if (!ptx::mbar_wait(ofull_bar(stage), phase, abort_flag)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t a = sbase + 64 * 1024 + stage * 2 * kTile16;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * kTile8 + (kk & 3) * 32;
              ptx::mma_f16(d_tmem, ptx::sdesc_sw128(a + off), ptx::sdesc_sw128(a + kTile16 + off), idesc,
                           (kb | kk) != 0);
            }
            ptx::mma_commit(oempty_bar(stage));
            if (++stage == 2) { stage = 0; phase ^= 1u; }
          } else {
            if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t a = sbase + stage * 2 * kTile8;
            const uint64_t adesc = ptx::sdesc_sw128(a), bdesc = ptx::sdesc_sw128(a + kTile8);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) ptx::mma_f8(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
            ptx::mma_commit(empty_bar(stage));
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
          }
        }
        if (ok) ptx::mma_commit(tfull_bar(b));
      }
      ptx::mma_commit(done_bar);
      ptx::mbar_wait_drain(done_bar, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-3)
    const int r = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    for (int it = 0;; ++it) {
      const int t = next_task(it);
      if (t < 0 || t >= num_tasks) break;
      const Task k = decode_task(args, n_tiles, t);
      const int b = it & 1;
      if (!ptx::mbar_wait(tfull_bar(b), (it >> 1) & 1, abort_flag)) break;
      ptx::tc_fence_after();
      const bool valid = r < k.rows;
      const int row = k.row0 + r;
      const float sx = valid ? __ldg(args.sx + row) : 0.f;
      const float* swp = args.sw + static_cast<size_t>(k.e) * args.N + k.nt * kLBN;
#pragma unroll 1
      for (int cc = 0; cc < kLBN / 32; ++cc) {
        uint32_t d[32];
        ptx::tmem_ld32(tmem_base + lane_off + b * kLBN + cc * 32, d);
        ptx::tmem_ld_wait();
        if (valid) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 s4 = __ldg(reinterpret_cast<const float4*>(swp + cc * 32 + j));
            v[j] = sx * s4.x * __uint_as_float(d[j]);
            v[j + 1] = sx * s4.y * __uint_as_float(d[j + 1]);
            v[j + 2] = sx * s4.z * __uint_as_float(d[j + 2]);
            v[j + 3] = sx * s4.w * __uint_as_float(d[j + 3]);
          }
          const size_t o = static_cast<size_t>(row) * args.N + k.nt * kLBN + cc * 32;
          if (args.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(args.out) + o);
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) + o);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pack_bf16(v[8 * j], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                                  pack_bf16(v[8 * j + 4], v[8 * j + 5]), pack_bf16(v[8 * j + 6], v[8 * j + 7]));
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
  if (warp == 5) ptx::tmem_dealloc(tmem_base, kLTmemCols);
  if (tid == 0 && *abort_flag) report_error(args.err, MOE_DEVERR_TIMEOUT);
}

}  // namespace

size_t lowp_workspace_bytes(int E) { return kWsHeader + align_up(static_cast<size_t>(E + 1) * 4, 256); }

}  // namespace moe

extern "C" size_t gmm_lowp_workspace_size(int M, int K, int N, int E) {
  (void)M; (void)K; (void)N;
  if (E <= 0) return 0;
  return moe::lowp_workspace_bytes(E);
}

extern "C" moe_status_t gmm_lowp(const void* input, const void* weights, const float* scales_x,
                                 const float* scales_w, const int32_t* expert_offsets, const int32_t* expert_sizes,
                                 void* out, int M, int K, int N, int E, int in_dt, int out_dt, void* ws,
                                 size_t ws_bytes, void* stream) {
  using namespace moe;
  if (M < 0 || K <= 0 || N <= 0 || E < 1 || E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (in_dt != MOE_DT_I8 && in_dt != MOE_DT_E4M3) return MOE_ERR_INVALID_ARG;
  if (out_dt != MOE_DT_BF16 && out_dt != MOE_DT_F32) return MOE_ERR_INVALID_ARG;
  if (!weights || !scales_w || !expert_offsets || !expert_sizes) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!input || !scales_x || !out)) return MOE_ERR_INVALID_ARG;
  if (K % kLBK != 0 || N % kLBN != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(input) || !aligned16(weights) || !aligned16(scales_w) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(E) * N >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < lowp_workspace_bytes(E) || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  if (M == 0) return MOE_OK;
  cudaStream_t s = as_stream(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(w);
  int* counter = reinterpret_cast<int*>(w + 4);
  int* num_tasks = reinterpret_cast<int*>(w + 8);
  int32_t* mt_prefix = reinterpret_cast<int32_t*>(w + kWsHeader);
  const int n_tiles = N / kLBN;
  lowp_prep_kernel<<<1, 1024, 0, s>>>(expert_offsets, expert_sizes, E, M, n_tiles, mt_prefix, counter, num_tasks,
                                      err);
  moe_status_t st = launch_status();
  if (st != MOE_OK) return st;
  const bool i8 = in_dt == MOE_DT_I8;
  CUtensorMap map_x, map_w;
  if (!make_tmap_u8_2d(&map_x, input, M, K, !i8)) return MOE_ERR_CUDA;
  if (!make_tmap_u8_2d(&map_w, weights, static_cast<uint64_t>(E) * N, K, !i8)) return MOE_ERR_CUDA;
  LowpArgs a{};
  a.sx = scales_x; a.sw = scales_w; a.offsets = expert_offsets; a.sizes = expert_sizes; a.mt_prefix = mt_prefix;
  a.counter = counter; a.num_tasks = num_tasks; a.out = out; a.err = err;
  a.M = M; a.K = K; a.N = N; a.E = E; a.out_f32 = out_dt == MOE_DT_F32;
  const void* fn = i8 ? reinterpret_cast<const void*>(gmm_lowp_kernel<true>)
                      : reinterpret_cast<const void*>(gmm_lowp_kernel<false>);
  if (!ensure_smem_attr(fn, static_cast<int>(kLSmem))) return MOE_ERR_CUDA;
  if (i8)
    gmm_lowp_kernel<true><<<num_sms(), kLThreads, kLSmem, s>>>(map_x, map_w, a);
  else
    gmm_lowp_kernel<false><<<num_sms(), kLThreads, kLSmem, s>>>(map_x, map_w, a);
  return launch_status();
}
