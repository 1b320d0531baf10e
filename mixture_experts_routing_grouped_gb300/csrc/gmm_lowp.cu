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
// tcgen05 has no integer MMA on sm_103a, so INT8 codes are widened to fp16
// (exact for |q| <= 128) and the MMA is kind::f16 with fp32 accumulation: the
// activation codes once, by a pre-pass into the workspace (every row block is
// reused by all N / 128 column blocks, so widening it per tile repeated the work
// N / 128 times and bounded the kernel), the weight codes per tile by eight
// converter warps, which read the codes TMA brought into shared memory and
// write the fp16 values straight into tensor memory. The MMA takes the widened
// weights as its A operand from tensor memory and the widened activations as
// its B operand from shared memory, so the product is transposed (accumulator
// lane = output channel, column = token) and its token count N is the task's
// row count rounded up to 16: an expert with 60 rows costs a 128 x 64 MMA, and
// only the 32-row slabs holding its rows are loaded. Staging the widened
// weights through shared memory instead cost the MMA a second 32 KB operand
// read and the converters a 32 KB write per K step, and shared-memory
// bandwidth bounded the kernel.
//
// Kernel shape (one persistent CTA per SM): warps 0-3 epilogue, warp 4 TMA
// producer (FP8: both operands; INT8: weight codes), warp 5
// owner of TMEM + MMA issuer, INT8 only: warps 6-13 weight converters, warp 14
// TMA producer of the widened activations; then four more epilogue warps (the
// first four drain accumulator columns 0-63, these 64-127) and the task
// scheduler, which claims and decodes tasks for the others. Tile 128 rows x
// 128 columns x 128 K; a task is (expert, 128-row block, 128-column block),
// ordered expert, column block, row block so that CTAs running together share
// each weight tile in L2. Rows of a block past the expert's end are computed on
// whatever TMA brought (the next expert's rows or zero fill) and never stored.
#include "common.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <cuda_fp16.h>

namespace moe {

bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, bool swizzle128);
bool make_tmap_bf16_2d_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, int box_rows);

namespace {

constexpr int kLBM = 128, kLBN = 128, kLBK = 128;      // K in elements (= bytes for 8-bit codes)
constexpr int kTile8 = kLBM * kLBK;                     // 16 KB: one 8-bit operand tile
constexpr int kF8Stages = 7;                            // fp8: 7 x (A 16 KB + B 16 KB)
constexpr int kTile16 = kLBM * kLBK * 2;                // 32 KB: one fp16 operand tile (2 column blocks)
constexpr int kI8BStages = 6;                           // int8: 6 x 16 KB weight codes
constexpr int kI8AStages = 4;                           // int8: 4 x 32 KB widened activations
constexpr int kI8Ops = 4;                               // int8: widened weight tiles in TMEM, 64 columns each
constexpr int kI8ConvWarps = 8;
constexpr int kI8AWarp = 6 + kI8ConvWarps;              // warp 14: activation producer
constexpr int kI8AOff = kI8BStages * kTile8;
constexpr int kI8Slab = 32;                             // int8: activation rows per TMA load
constexpr int kQ = 4;                                   // task queue slots
constexpr int kI8OpCol = 2 * kLBN;                      // int8: first TMEM column of the weight tiles
template <bool I8>
constexpr int lowp_tmem_cols() { return I8 ? 512 : 2 * kLBN; }  // accumulators (+ int8 weight tiles)
static_assert(kI8OpCol + kI8Ops * kLBK / 2 <= 512, "tensor memory columns");
constexpr int kF8Ring = kF8Stages * 2 * kTile8;         // 224 KB
constexpr int kI8Ring = kI8AOff + kI8AStages * kTile16; // 224 KB
constexpr size_t kLSmem = 1024 + kI8Ring + 512 + 2 * kLBN * 4 + kQ * 16;
static_assert(kLSmem <= 232448, "shared memory per CTA");
template <bool I8>
constexpr int lowp_threads() { return 32 * ((I8 ? kI8AWarp + 1 : 6) + 5); }  // + 4 more epilogue warps + scheduler
// The second half of the epilogue: four warps after the kernel's other roles.
template <bool I8>
constexpr int lowp_epi2_warp0() { return I8 ? kI8AWarp + 1 : 6; }
// The task scheduler: the last warp.
template <bool I8>
constexpr int lowp_sched_warp() { return lowp_epi2_warp0<I8>() + 4; }

struct LowpArgs {
  const float* sx;
  const float* sw;
  const int32_t* offsets;
  const int32_t* sizes;
  int* counter;              // tasks claimed beyond the first gridDim.x (zero at launch)
  int* exit_ticket;          // CTAs finished (zero at launch); the last one re-zeroes both
  void* out;
  int* err;
  int M, K, N, E, out_f32;
};

// A task: expert e's 128-row block starting at row0 (rows of them real) times column
// block nt. Task ids run expert by expert; within an expert, column block by column
// block, row blocks fastest, so that CTAs running together share each weight tile in
// L2. Expert e's tasks are [P[e] * n_tiles, P[e+1] * n_tiles), P the prefix sum of the
// experts' row-block counts (experts with inconsistent metadata count zero blocks).
struct Task {
  int e, row0, rows, nt;
};

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

// INT8 activation codes -> fp16 (exact), 16 codes per thread and step.
__global__ void __launch_bounds__(256) widen_i8_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                       size_t n16) {
  pdl_trigger();
  pdl_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(src + i);
    uint32_t h[8];
    i8x4_to_f16x4(v.x, h[0], h[1]);
    i8x4_to_f16x4(v.y, h[2], h[3]);
    i8x4_to_f16x4(v.z, h[4], h[5]);
    i8x4_to_f16x4(v.w, h[6], h[7]);
    dst[2 * i] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[2 * i + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

template <bool I8>
__global__ void __launch_bounds__(lowp_threads<I8>(), 1)
    gmm_lowp_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                    const LowpArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  constexpr int kStages = I8 ? kI8BStages : kF8Stages;
  // fp8: stage s = [A 16 KB | B 16 KB] at s*32 KB.
  // int8: weight-code stage s (16 KB: [128 rows][128 B], 128B swizzle) at s*16 KB;
  //       widened activations a (32 KB: 2 column blocks of [128 rows][128 B],
  //       128B swizzle) after the code ring. Widened weight tile o sits in TMEM
  //       columns [kI8OpCol + 64 o, +64): lane = channel, two K values a column.
  uint8_t* ctl = smem + (I8 ? kI8Ring : kF8Ring);
  const uint32_t bar0 = ptx::smem_u32(ctl);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };                 // staging / stage landed
  auto empty_bar = [&](int s) { return bar0 + 8u * (8 + s); };          // staging / stage free
  auto ofull_bar = [&](int s) { return bar0 + 8u * (16 + s); };         // int8: fp16 weight tile ready
  auto oempty_bar = [&](int s) { return bar0 + 8u * (20 + s); };        // int8: fp16 weight tile free
  auto tfull_bar = [&](int b) { return bar0 + 8u * (24 + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (26 + b); };
  auto qfull_bar = [&](int q) { return bar0 + 8u * (28 + q); };
  auto qempty_bar = [&](int q) { return bar0 + 8u * (32 + q); };
  const uint32_t done_bar = bar0 + 8u * 36;
  auto afull_bar = [&](int s) { return bar0 + 8u * (37 + s); };         // int8: activations landed
  auto aempty_bar = [&](int s) { return bar0 + 8u * (41 + s); };        // int8: activations free
  auto taken_bar = [&](int q) { return bar0 + 8u * (45 + q); };         // queue entry taken by the TMA thread
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + 400);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl + 404);
  float* scl = reinterpret_cast<float*>(ctl + 512);  // [2][128] epilogue scales: fp8 channel, int8 token
  volatile int* tq = reinterpret_cast<volatile int*>(ctl + 512 + 2 * kLBN * 4);  // [kQ][4] claimed tasks

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  const int n_tiles = args.N / kLBN;
  const int kblocks = args.K / kLBK;
  constexpr int kConvThreads = I8 ? 32 * kI8ConvWarps : 0;
  constexpr int kConsumers = 1 + 1 + 256 + kConvThreads + (I8 ? 1 : 0);  // TMA, MMA, epilogue, int8 roles
  constexpr int kEpi2 = lowp_epi2_warp0<I8>();

  if (tid == 0) {
    for (int s = 0; s < 8; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), I8 ? kConvThreads : 1);  // int8: released by the converters
    }
    for (int s = 0; s < kI8AStages; ++s) {
      ptx::mbar_init(afull_bar(s), 1);
      ptx::mbar_init(aempty_bar(s), 1);
    }
    for (int s = 0; s < 4; ++s) {
      ptx::mbar_init(ofull_bar(s), kConvThreads > 0 ? kConvThreads : 1);
      ptx::mbar_init(oempty_bar(s), 1);
      ptx::mbar_init(qfull_bar(s), 1);
      ptx::mbar_init(qempty_bar(s), kConsumers);
    }
    for (int q = 0; q < kQ; ++q) ptx::mbar_init(taken_bar(q), 1);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), 256);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), lowp_tmem_cols<I8>());
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a programmatic dependent of the kernel before it in the stream (for
  // INT8 the activation widening): the prologue above overlapped that kernel; nothing
  // in global memory is read or written before it has completed.
  pdl_wait();

  // Task queue consumer: the claiming thread decodes every task once and publishes
  // it whole, so that no consumer waits on the dependent global loads of a decode.
  // Returns false when the tasks are done (expert -1) or on abort.
  auto next_task = [&](int it, Task& k) -> bool {
    const int q = it % kQ;
    if (!ptx::mbar_wait(qfull_bar(q), (static_cast<uint32_t>(it / kQ) & 1u), abort_flag)) return false;
    k.e = tq[4 * q];
    k.row0 = tq[4 * q + 1];
    k.rows = tq[4 * q + 2];
    k.nt = tq[4 * q + 3];
    ptx::mbar_arrive(qempty_bar(q));
    return k.e >= 0;
  };

  if (warp == lowp_sched_warp<I8>()) {
    // ------------------------------------------------------------ task scheduler
    // The CTA's first task is blockIdx.x; every further one is claimed from the global
    // counter (an L2 round trip) once the TMA thread has taken the previous one, so a
    // CTA holds at most one task beyond the one it is loading and the claims stay
    // balanced to the end. The whole warp decodes: it walks the experts 32 at a time
    // (lane l holds expert c0 + l's offset, size, 128-row block count and the
    // inclusive prefix of the counts), which it can do forwards only because a CTA's
    // claims increase. Experts whose metadata do not add up count zero blocks and set
    // MOE_DEVERR_GROUP_META (every CTA walks every expert by the time the tasks run out).
    // Claiming and decoding in the TMA thread stalled its loads at every task boundary
    // by a chain of dependent global loads; with small K a task is only a few K steps
    // (the article's small-K case, section 4.2, interleaves two experts per block
    // against the same gap).
    int c0 = 0, base = 0;  // first expert of the chunk, row blocks before it
    int o_l = 0, s_l = 0, nb_l = 0, incl_l = 0, total = 0;
    auto load_chunk = [&]() {
      const int e = c0 + lane;
      o_l = 0; s_l = 0; nb_l = 0;
      if (e < args.E) {
        o_l = __ldg(args.offsets + e);
        const int o1 = __ldg(args.offsets + e + 1);
        s_l = __ldg(args.sizes + e);
        if (s_l >= 0 && o_l >= 0 && o1 <= args.M && o1 - o_l == s_l) nb_l = (s_l + kLBM - 1) / kLBM;
        else report_error(args.err, MOE_DEVERR_GROUP_META);
      }
      incl_l = nb_l;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl_l, o);
        if (lane >= o) incl_l += v;
      }
      total = __shfl_sync(0xffffffffu, incl_l, 31);
    };
    if (blockIdx.x == 0 && lane == 0 &&
        (__ldg(args.offsets) != 0 || __ldg(args.offsets + args.E) != args.M))
      report_error(args.err, MOE_DEVERR_GROUP_META);
    load_chunk();
    for (int it = 0;; ++it) {
      if (it > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(taken_bar((it - 1) % kQ),
                                                             static_cast<uint32_t>((it - 1) / kQ) & 1u, abort_flag)))
        break;
      int t = static_cast<int>(blockIdx.x);
      if (it > 0 && lane == 0) t = static_cast<int>(gridDim.x) + atomicAdd(args.counter, 1);
      t = __shfl_sync(0xffffffffu, t, 0);
      const int mb = t / n_tiles;  // expert e holds the task iff P[e] <= mb < P[e + 1]
      Task k;
      k.e = -1; k.row0 = 0; k.rows = 0; k.nt = 0;
      while (c0 < args.E) {
        const unsigned m = __ballot_sync(0xffffffffu, c0 + lane < args.E && base + incl_l > mb);
        if (m != 0u) {
          const int l = __ffs(m) - 1;
          const int pe = base + __shfl_sync(0xffffffffu, incl_l - nb_l, l);
          const int mcount = __shfl_sync(0xffffffffu, nb_l, l);
          const int off = __shfl_sync(0xffffffffu, o_l, l);
          const int size = __shfl_sync(0xffffffffu, s_l, l);
          const int local = t - pe * n_tiles;
          k.e = c0 + l;
          k.nt = local / mcount;
          k.row0 = off + (local - k.nt * mcount) * kLBM;
          k.rows = min(kLBM, off + size - k.row0);
          break;
        }
        base += total;
        c0 += 32;
        load_chunk();
      }
      if (lane == 0) {
        const int q = it % kQ;
        if (ptx::mbar_wait(qempty_bar(q), (static_cast<uint32_t>(it / kQ) & 1u) ^ 1u, abort_flag)) {
          tq[4 * q] = k.e;
          tq[4 * q + 1] = k.row0;
          tq[4 * q + 2] = k.rows;
          tq[4 * q + 3] = k.nt;
          ptx::mbar_arrive(qfull_bar(q));
        } else {
          k.e = -1;
        }
      }
      if (__shfl_sync(0xffffffffu, k.e, 0) < 0) break;
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        Task k;
        if (!next_task(it, k)) break;
        ptx::mbar_arrive(taken_bar(it % kQ));
        const int wrow = k.e * args.N + k.nt * kLBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          if constexpr (I8) {
            const uint32_t dst = sbase + stage * kTile8;  // weight codes
            ptx::mbar_arrive_expect_tx(full_bar(stage), kTile8);
            ptx::tma_load_2d(dst, &map_w, full_bar(stage), kb * kLBK, wrow);
          } else {
            const uint32_t dst = sbase + stage * 2 * kTile8;
            ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * kTile8);
            ptx::tma_load_2d(dst, &map_x, full_bar(stage), kb * kLBK, k.row0);
            ptx::tma_load_2d(dst + kTile8, &map_w, full_bar(stage), kb * kLBK, wrow);
          }
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
#pragma unroll
      for (int s = 0; s < kStages; ++s) {
        const int fills = issued / kStages + (s < issued % kStages ? 1 : 0);
        if (fills > 0) ptx::mbar_wait_drain(full_bar(s), (fills - 1) & 1);
      }
    }
    __syncwarp();
  } else if (I8 && warp == kI8AWarp) {
    // ------------------------------------------------------------ int8: widened-activation producer
    if (lane == 0) {
      int astage = 0, issued = 0;
      uint32_t aphase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        Task k;
        if (!next_task(it, k)) break;
        const int slabs = (k.rows + kI8Slab - 1) / kI8Slab;  // only the 32-row slabs holding the task's rows
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(aempty_bar(astage), aphase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t dst = sbase + kI8AOff + astage * kTile16;
          ptx::mbar_arrive_expect_tx(afull_bar(astage), slabs * kI8Slab * 128 * 2);
          for (int j = 0; j < slabs; ++j) {
            const uint32_t o = j * kI8Slab * 128;
            ptx::tma_load_2d(dst + o, &map_x, afull_bar(astage), kb * kLBK, k.row0 + j * kI8Slab);
            ptx::tma_load_2d(dst + kTile8 + o, &map_x, afull_bar(astage), kb * kLBK + kLBK / 2,
                             k.row0 + j * kI8Slab);
          }
          ++issued;
          if (++astage == kI8AStages) { astage = 0; aphase ^= 1u; }
        }
      }
#pragma unroll
      for (int st = 0; st < kI8AStages; ++st) {
        const int fills = issued / kI8AStages + (st < issued % kI8AStages ? 1 : 0);
        if (fills > 0) ptx::mbar_wait_drain(afull_bar(st), (fills - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp >= 6 && warp < kEpi2) {
    // ------------------------------------------------------------ int8 -> fp16 weight converters
    if constexpr (I8) {
      // Thread = one weight row (channel r, the TMEM lane this warp may write) and one half
      // of the K step: codes [64 half, +64) of row r, four 16-byte chunks of the swizzled
      // stage (chunk j of row r sits at chunk j ^ (r & 7), so a warp's loads spread over all
      // banks), widened to 32 words of fp16 pairs and stored to TMEM columns [32 half, +32)
      // of the weight tile.
      const int quarter = warp & 3;
      const int half = (warp - 6) >> 2;
      const int r = quarter * 32 + lane;
      const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
      int stage = 0, ostage = 0;
      uint32_t phase = 0, ophase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        Task k;
        if (!__all_sync(0xffffffffu, next_task(it, k))) break;  // the warp goes on, or leaves, as one
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(full_bar(stage), phase, abort_flag))) { ok = false; break; }
          const uint8_t* src = smem + stage * kTile8 + r * 128;
          uint4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            v[q] = *reinterpret_cast<const uint4*>(src + ((((half << 2) + q) ^ (r & 7)) << 4));
          uint32_t h[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            i8x4_to_f16x4(v[q].x, h[8 * q + 0], h[8 * q + 1]);
            i8x4_to_f16x4(v[q].y, h[8 * q + 2], h[8 * q + 3]);
            i8x4_to_f16x4(v[q].z, h[8 * q + 4], h[8 * q + 5]);
            i8x4_to_f16x4(v[q].w, h[8 * q + 6], h[8 * q + 7]);
          }
          ptx::mbar_arrive(empty_bar(stage));
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(oempty_bar(ostage), ophase ^ 1u, abort_flag))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          ptx::tmem_st32(tmem_base + lane_off + kI8OpCol + ostage * (kLBK / 2) + half * 32, h);
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          ptx::mbar_arrive(ofull_bar(ostage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
          if (++ostage == kI8Ops) { ostage = 0; ophase ^= 1u; }
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (ptx::elect_one()) {
      const uint32_t idesc = I8 ? (ptx::idesc_bf16_f32(kLBM, kLBN) & ~((7u << 7) | (7u << 10)))  // fp16 A/B
                                : ptx::idesc_e4m3_f32(kLBM, kLBN);
      int stage = 0, ostage = 0, astage = 0;
      uint32_t phase = 0, ophase = 0, aphase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        Task k;
        if (!next_task(it, k)) break;
        uint32_t idesc_t = idesc;
        if constexpr (I8) {  // transposed product: N = the task's tokens, rounded up to 16
          const int n_tok = (k.rows + 15) & ~15;
          idesc_t = (idesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(n_tok >> 3) << 17);
        }
        const int b = it & 1;
        if (!ptx::mbar_wait(tempty_bar(b), ((it >> 1) & 1) ^ 1u, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kLBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if constexpr (I8) {
            if (!ptx::mbar_wait(afull_bar(astage), aphase, abort_flag) ||
                !ptx::mbar_wait(ofull_bar(ostage), ophase, abort_flag)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t act = sbase + kI8AOff + astage * kTile16;
            const uint32_t wt = tmem_base + kI8OpCol + ostage * (kLBK / 2);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // K 16 kk .. +16: 8 TMEM columns, 32 bytes of a 128-byte row
              const uint32_t off = (kk >> 2) * kTile8 + (kk & 3) * 32;
              ptx::mma_f16_ts(d_tmem, wt + 8 * kk, ptx::sdesc_sw128(act + off), idesc_t, (kb | kk) != 0);
            }
            ptx::mma_commit(oempty_bar(ostage));
            ptx::mma_commit(aempty_bar(astage));
            if (++ostage == kI8Ops) { ostage = 0; ophase ^= 1u; }
            if (++astage == kI8AStages) { astage = 0; aphase ^= 1u; }
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
    // ------------------------------------------------------------ epilogue (warps 0-3 and kEpi2..kEpi2+3)
    // Two warps per TMEM lane quarter, each draining half of the tile's columns. The scales that
    // vary along the columns (fp8: the tile's 128 channel scales; int8, transposed: its tokens'
    // scales) are copied to shared memory (one per thread of the first four warps, double
    // buffered by accumulator) before the wait for the accumulator, so that no global load sits
    // between a TMEM chunk and its stores; each chunk's TMEM load is issued before the previous
    // chunk is scaled and stored.
    const bool second = warp >= kEpi2;
    const int quarter = warp & 3;  // a warp reaches only TMEM lanes [32 * (warp % 4), +32)
    const int c0 = second ? kLBN / 64 : 0;  // first 32-column chunk of this warp (two chunks each)
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    if constexpr (I8) {
      // Lane r holds output channel nt * 128 + r; column m holds the task's token m. A warp's
      // store for one token writes 32 consecutive channels of its output row.
      for (int it = 0;; ++it) {
        Task k;
        const bool got = next_task(it, k);
        const int b = it & 1;
        float* sc = scl + b * kLBN;
        float sw = 0.f;
        if (got) {
          if (!second) sc[r] = r < k.rows ? __ldg(args.sx + k.row0 + r) : 0.f;
          sw = __ldg(args.sw + static_cast<size_t>(k.e) * args.N + k.nt * kLBN + r);
        }
        // the eight epilogue warps: scales staged; they leave the loop together (they meet
        // at this named barrier every task)
        if (ptx::bar_any(1, 256, !got)) break;
        const int chunks = min(kLBN / 64, max(0, (k.rows - c0 * 32 + 31) / 32));  // warp-uniform
        const bool full = ptx::mbar_wait(tfull_bar(b), (it >> 1) & 1, abort_flag);
        if (ptx::bar_any(1, 256, !full)) break;
        ptx::tc_fence_after();
        uint32_t d[2][32];
        if (chunks > 0) ptx::tmem_ld32(tmem_base + lane_off + b * kLBN + c0 * 32, d[0]);
#pragma unroll
        for (int ci = 0; ci < kLBN / 64; ++ci) {
          if (ci >= chunks) break;
          const int cc = c0 + ci;
          ptx::tmem_ld_wait();
          if (ci + 1 < chunks) ptx::tmem_ld32(tmem_base + lane_off + b * kLBN + (cc + 1) * 32, d[(ci + 1) & 1]);
          const uint32_t* dc = d[ci & 1];
          const int m_end = min(32, k.rows - cc * 32);
          const size_t o = static_cast<size_t>(k.row0 + cc * 32) * args.N + k.nt * kLBN + r;
          if (args.out_f32) {
            float* dst = static_cast<float*>(args.out) + o;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < m_end) dst[static_cast<size_t>(j) * args.N] = sc[cc * 32 + j] * sw * __uint_as_float(dc[j]);
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(args.out) + o;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < m_end)
                dst[static_cast<size_t>(j) * args.N] = __float2bfloat16_rn(sc[cc * 32 + j] * sw * __uint_as_float(dc[j]));
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(tempty_bar(b));
      }
    } else {
    for (int it = 0;; ++it) {
      Task k;
      const bool got = next_task(it, k);
      const int b = it & 1;
      float* sc = scl + b * kLBN;
      const bool valid = got && r < k.rows;
      const int row = k.row0 + r;
      float sx = 0.f;
      if (got) {
        if (!second) sc[r] = __ldg(args.sw + static_cast<size_t>(k.e) * args.N + k.nt * kLBN + r);
        if (valid) sx = __ldg(args.sx + row);
      }
      // the eight epilogue warps: scales staged; they leave the loop together (they meet
      // at this named barrier every task)
      if (ptx::bar_any(1, 256, !got)) break;
      const bool full = ptx::mbar_wait(tfull_bar(b), (it >> 1) & 1, abort_flag);
      if (ptx::bar_any(1, 256, !full)) break;
      ptx::tc_fence_after();
      uint32_t d[2][32];
      ptx::tmem_ld32(tmem_base + lane_off + b * kLBN + c0 * 32, d[0]);
#pragma unroll
      for (int ci = 0; ci < kLBN / 64; ++ci) {
        const int cc = c0 + ci;
        ptx::tmem_ld_wait();
        if (ci + 1 < kLBN / 64) ptx::tmem_ld32(tmem_base + lane_off + b * kLBN + (cc + 1) * 32, d[(ci + 1) & 1]);
        if (valid) {
          const uint32_t* dc = d[ci & 1];
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 s4 = *reinterpret_cast<const float4*>(sc + cc * 32 + j);
            v[j] = sx * s4.x * __uint_as_float(dc[j]);
            v[j + 1] = sx * s4.y * __uint_as_float(dc[j + 1]);
            v[j + 2] = sx * s4.z * __uint_as_float(dc[j + 2]);
            v[j + 3] = sx * s4.w * __uint_as_float(dc[j + 3]);
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
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 5) ptx::tmem_dealloc(tmem_base, lowp_tmem_cols<I8>());
  if (tid == 0) {
    if (*abort_flag) report_error(args.err, MOE_DEVERR_TIMEOUT);
    // Every claim of this CTA has returned (the barrier above); the last CTA out
    // leaves both counters zero for the next call on this workspace.
    __threadfence();
    if (atomicAdd(args.exit_ticket, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(args.counter, 0);
      atomicExch(args.exit_ticket, 0);
    }
  }
}

}  // namespace

// Header (error word, task counter, exit ticket), then (INT8 inputs) the fp16 copy of the
// activation codes.
size_t lowp_meta_bytes(int E) {
  (void)E;
  return kWsHeader;
}
size_t lowp_workspace_bytes(int M, int K, int E) {
  return lowp_meta_bytes(E) + align_up(static_cast<size_t>(M) * K * 2, 256);
}

}  // namespace moe

extern "C" size_t gmm_lowp_workspace_size(int M, int K, int N, int E) {
  (void)N;
  if (E <= 0 || M < 0 || K < 0) return 0;
  return moe::lowp_workspace_bytes(M, K, E);
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
  const bool i8 = in_dt == MOE_DT_I8;
  const size_t need = i8 ? lowp_workspace_bytes(M, K, E) : lowp_meta_bytes(E);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  if (M == 0) return MOE_OK;
  cudaStream_t s = as_stream(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(w);
  int* counter = reinterpret_cast<int*>(w + 4);
  int* exit_ticket = reinterpret_cast<int*>(w + 8);
  moe_status_t st = MOE_OK;
  CUtensorMap map_x, map_w;
  if (i8) {
    // widen the activation codes once; the kernel loads them as fp16 tiles (a
    // 2-byte tensor map: TMA moves bytes, the bf16 element type only sizes them)
    void* xh = w + lowp_meta_bytes(E);
    const size_t n16 = static_cast<size_t>(M) * K / 16;
    const int grid = static_cast<int>(std::min<size_t>((n16 + 255) / 256, static_cast<size_t>(num_sms()) * 8));
    st = launch_pdl(widen_i8_kernel, dim3(grid), dim3(256), 0, s, static_cast<const uint4*>(input),
                    static_cast<uint4*>(xh), n16);
    if (st != MOE_OK) return st;
    if (!make_tmap_bf16_2d_rows(&map_x, xh, M, K, kI8Slab)) return MOE_ERR_CUDA;
  } else if (!make_tmap_u8_2d(&map_x, input, M, K, true)) {
    return MOE_ERR_CUDA;
  }
  if (!make_tmap_u8_2d(&map_w, weights, static_cast<uint64_t>(E) * N, K, true)) return MOE_ERR_CUDA;
  LowpArgs a{};
  a.sx = scales_x; a.sw = scales_w; a.offsets = expert_offsets; a.sizes = expert_sizes;
  a.counter = counter; a.exit_ticket = exit_ticket; a.out = out; a.err = err;
  a.M = M; a.K = K; a.N = N; a.E = E; a.out_f32 = out_dt == MOE_DT_F32;
  const void* fn = i8 ? reinterpret_cast<const void*>(gmm_lowp_kernel<true>)
                      : reinterpret_cast<const void*>(gmm_lowp_kernel<false>);
  if (!ensure_smem_attr(fn, static_cast<int>(kLSmem))) return MOE_ERR_CUDA;
  if (i8)
    return launch_pdl(gmm_lowp_kernel<true>, dim3(num_sms()), dim3(lowp_threads<true>()), kLSmem, s, map_x, map_w, a);
  return launch_pdl(gmm_lowp_kernel<false>, dim3(num_sms()), dim3(lowp_threads<false>()), kLSmem, s, map_x, map_w, a);
}
