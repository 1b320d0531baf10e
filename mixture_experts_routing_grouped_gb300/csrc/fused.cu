// moe_fused_forward: the routed MoE layer on one stream.
//
// Follows the mini-sglang MoE chapter, FusedMoeBackend.forward: routing
// (select_experts, here the grouped top-k), moe_align_block_size, the gate_up
// grouped GEMM (rows gathered as pair / topk), silu(gate) * up, the down grouped
// GEMM multiplied by the route weight, and the sum over the topk slots of every
// token. The page's intermediate buffers cache1..cache3 ([T*k, 2I], [T*k, I],
// [T*k, H]) are replaced by h = silu(gate) * up in sorted order (written once by
// the gate_up epilogue, read once by the down GEMM) and an fp32 [T, H]
// accumulator that the down epilogue adds into; the page's host synchronisation
// on the padded length is replaced by a device-side length read by the GEMMs.
#include "common.cuh"

namespace moe {

moe_status_t validate_routing(int T, int E, int G, int kg, int k, int scoring);
moe_status_t launch_grouped_topk(const float* gating, int T, int E, int G, int kg, int k, int scoring, int renorm,
                                 float rsf, float* w, int32_t* ids, cudaStream_t s, float* zero_rows, int zero_cols,
                                 int* zero_cnt, int cnt_per_row);
moe_status_t launch_grouped_topk_tile_hist(const float* gating, int T, int E, int G, int kg, int k, int scoring,
                                           int renorm, float rsf, float* w, int32_t* ids, int32_t* tile_hist,
                                           int* err, float* zero_rows, int zero_cols, int* rows_out,
                                           int* tokens_per_row, cudaStream_t s);
int route_hist_rows(int T, int E, int G, int kg, int k, const void* w, const void* ids, bool zero_rows,
                    int* tokens_per_row);
size_t align_tile_hist_bytes(int T, int E);
bool align_takes_tile_hists(int num_pairs, int E, int tile_rows, int pairs_per_tile);
moe_status_t launch_align_from_tile_hists(const int32_t* ids, int num_pairs, int E, int block_m,
                                          int32_t* sorted_ids, int32_t* expert_ids, int32_t* expert_offsets,
                                          int32_t* ntpp, const int32_t* tile_hist, int tile_rows,
                                          int pairs_per_tile, cudaStream_t s, int32_t* sorted_tok, int topk,
                                          int* zero_word);
size_t align_max_padded(int num_pairs, int E, int block_m);
size_t align_scratch_bytes(int num_pairs, int E);
moe_status_t launch_align(const int32_t* ids, int num_pairs, int E, int block_m, int32_t* sorted_ids,
                          int32_t* expert_ids, int32_t* expert_offsets, int32_t* ntpp, void* scratch, int* err,
                          cudaStream_t s, int32_t* sorted_tok, int topk, int* zero_word);
moe_status_t launch_gemm_gate_up_pairs(const __nv_bfloat16* x, const __nv_bfloat16* w1, const int32_t* sorted_tok,
                                       const int32_t* offsets, __nv_bfloat16* h, int* err, int num_pairs, int topk,
                                       int H, int I, int E, float* y_clear, size_t y_clear_floats,
                                       int* tile_counter, cudaStream_t s);
moe_status_t launch_gemm_down(const __nv_bfloat16* h, const __nv_bfloat16* w2, const int32_t* sorted_ids,
                              const int32_t* expert_ids, const int32_t* ntpp, const float* topk_w, float* y_acc,
                              int* err, int num_pairs, int topk, int cap, int H, int I, int E, cudaStream_t s);

moe_status_t launch_gemm_gate_up_pairs_fp8(const uint8_t* qx, const float* sx, const uint8_t* w1, const float* sw1,
                                           const int32_t* sorted_tok, const int32_t* offsets, __nv_bfloat16* h,
                                           int* err, int H, int I, int E, float* y_clear, size_t y_clear_floats,
                                           int* tile_counter, cudaStream_t s);
moe_status_t launch_gemm_down_fp8(const uint8_t* qh, const float* sh, const uint8_t* w2, const float* sw2,
                                  const int32_t* sorted_ids, const int32_t* expert_ids, const int32_t* ntpp,
                                  const float* topk_w, float* y_acc, int* err, int num_pairs, int topk, int cap,
                                  int H, int I, int E, cudaStream_t s);
moe_status_t launch_quant_rows_e4m3_bf16(const __nv_bfloat16* x, int M, int K, uint8_t* q, float* s,
                                         const int* rows_dev, cudaStream_t st);

moe_status_t launch_swap_gate_up_fp8(const uint8_t* qx, const float* sx, const uint8_t* w1, const float* sw1,
                                     const int32_t* sorted_ids, const int32_t* offsets, __nv_bfloat16* h, int* err,
                                     int num_pairs, int topk, int H, int I, int E, cudaStream_t s);
moe_status_t launch_swap_down_fp8(const uint8_t* qh, const float* sh, const uint8_t* w2, const float* sw2,
                                  const int32_t* sorted_ids, const int32_t* offsets, const float* topk_w,
                                  float* y_acc, int* err, int num_pairs, int topk, int cap, int H, int I, int E,
                                  cudaStream_t s);
moe_status_t launch_swap_gate_up(const __nv_bfloat16* x, const __nv_bfloat16* w1, const int32_t* sorted_ids,
                                 const int32_t* offsets, __nv_bfloat16* h, int* err, int num_pairs, int topk, int H,
                                 int I, int E, int nmax, cudaStream_t s);
moe_status_t launch_swap_down(const __nv_bfloat16* h, const __nv_bfloat16* w2, const int32_t* sorted_ids,
                              const int32_t* offsets, const float* topk_w, float* y_acc, int* err, int num_pairs,
                              int topk, int cap, int H, int I, int E, int nmax, cudaStream_t s);

namespace {

// Kernel choice. Decode-sized problems (at most 32 rows per expert on average)
// use the swap-AB kernels with 16-row blocks and token tiles of <= 32; larger
// ones use the sorted-layout kernels with 128-row blocks.
struct Plan {
  bool swap;
  int nmax;
  int block_m;
};

Plan choose_plan(int T, int E, int topk) {
  Plan p{};
  const long long pairs = static_cast<long long>(T) * topk;
  if (pairs <= 32ll * E) {
    p.swap = true; p.nmax = 32; p.block_m = 16;
  } else {
    p.swap = false; p.nmax = 0; p.block_m = 128;
  }
  return p;
}

// y = bf16(y_acc): four independent 16-byte loads in flight per thread (one at a
// time left the kernel latency-bound on the just-written, L2-resident rows).
__global__ void __launch_bounds__(256) cast_f32_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                                            size_t n4) {
  pdl_trigger();
  pdl_wait();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4; i += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i + j * stride < n4) v[j] = src[i + j * stride];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (i + j * stride >= n4) break;
      const __nv_bfloat162 a = __floats2bfloat162_rn(v[j].x, v[j].y);
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[j].z, v[j].w);
      dst[i + j * stride] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
  }
}

struct FusedLayout {
  size_t align_scratch, sorted_ids, sorted_tok, expert_ids, expert_offsets, ntpp, h, y_acc, total;
  int cap;
};

FusedLayout fused_layout(int T, int H, int I, int E, int topk, int block_m) {
  FusedLayout L{};
  const int num_pairs = T * topk;
  L.cap = static_cast<int>(align_max_padded(num_pairs, E, block_m));
  size_t off = kWsHeader;
  const size_t own = align_scratch_bytes(num_pairs, E), tiles = align_tile_hist_bytes(T, E);
  L.align_scratch = off; off = align_up(off + (own > tiles ? own : tiles), 256);
  L.sorted_ids = off; off = align_up(off + static_cast<size_t>(L.cap) * 4, 256);
  L.sorted_tok = off; off = align_up(off + static_cast<size_t>(L.cap) * 4, 256);
  L.expert_ids = off; off = align_up(off + static_cast<size_t>(L.cap / block_m + 1) * 4, 256);
  L.expert_offsets = off; off = align_up(off + static_cast<size_t>(E + 1) * 4, 256);
  L.ntpp = off; off = align_up(off + 4, 1024);
  L.h = off; off = align_up(off + static_cast<size_t>(L.cap) * I * 2, 1024);
  L.y_acc = off; off = align_up(off + static_cast<size_t>(T) * H * 4, 256);
  L.total = off;
  return L;
}

// The FP8 forward's workspace: the bf16 forward's layout for the selected kernels, then
// the per-token e4m3 codes of x and their scales, then the per-row e4m3 codes of h and
// their scales.
struct Fp8Layout {
  FusedLayout base;
  size_t qx, sx, qh, sh, total;
};

Fp8Layout fp8_layout(int T, int H, int I, int E, int topk) {
  Fp8Layout L{};
  L.base = fused_layout(T, H, I, E, topk, choose_plan(T, E, topk).block_m);
  size_t off = align_up(L.base.total, 1024);
  L.qx = off; off = align_up(off + static_cast<size_t>(T) * H, 1024);
  L.sx = off; off = align_up(off + static_cast<size_t>(T) * 4, 1024);
  L.qh = off; off = align_up(off + static_cast<size_t>(L.base.cap) * I, 1024);
  L.sh = off; off = align_up(off + static_cast<size_t>(L.base.cap) * 4, 256);
  L.total = off;
  return L;
}

// A second stream per (host thread, device), with a fork and a join event, on which
// the FP8 forward quantises x while routing and align (small, latency-bound launches
// that leave most SMs idle) run on the caller's stream. Forked from and joined back
// into the caller's stream by events, so the call stays ordered on that stream and
// capturable into a CUDA graph. Created on first use and kept; null if creation
// failed (the work then stays on the caller's stream).
struct SideStream {
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool tried = false;
};

SideStream* side_stream() {
  constexpr int kMaxDevices = 64;
  thread_local SideStream per_device[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = per_device[dev];
  if (!ss.tried) {
    ss.tried = true;
    if (cudaStreamCreateWithFlags(&ss.st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      ss.st = nullptr;
    }
  }
  return ss.st ? &ss : nullptr;
}

thread_local cudaEvent_t g_stage_events[8];
thread_local int g_num_stage_events = 0;

inline void stage_mark(int i, cudaStream_t s) {
  if (i < g_num_stage_events) cudaEventRecord(g_stage_events[i], s);
}

int grid_for(size_t n4) {
  const size_t want = (n4 + 1023) / 1024;  // 256 threads x 4 elements
  const size_t cap = static_cast<size_t>(num_sms() > 0 ? num_sms() : 148) * 8;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

// Routing, then align, on stream s. Where the routing kernel for this shape can count the
// experts of its rows of tokens (the segmented and streaming kernels) and align can start
// from those counts, routing writes them into the align scratch and align skips its own
// counting pass (one launch fewer).
moe_status_t route_and_align(const float* gating, int T, int E, int G, int kg, int topk, int scoring, int renorm,
                             float rsf, float* topk_weights, int32_t* topk_ids, float* zero_rows, int zero_cols,
                             int block_m, int32_t* sorted_ids, int32_t* expert_ids, int32_t* offsets, int32_t* ntpp,
                             uint8_t* align_scratch, int* err, int32_t* sorted_tok, int* tile_counter,
                             cudaStream_t s) {
  const int num_pairs = T * topk;
  int32_t* tile_hist = reinterpret_cast<int32_t*>(align_scratch + 256);
  int tpr = 0;
  int rows = route_hist_rows(T, E, G, kg, topk, topk_weights, topk_ids, zero_rows != nullptr, &tpr);
  if (rows > 0 && !align_takes_tile_hists(num_pairs, E, rows, tpr * topk)) rows = 0;
  moe_status_t st;
  if (rows > 0) {
    int launched = 0;
    st = launch_grouped_topk_tile_hist(gating, T, E, G, kg, topk, scoring, renorm, rsf, topk_weights, topk_ids,
                                       tile_hist, err, zero_rows, zero_cols, &launched, &tpr, s);
    if (st != MOE_OK) return st;
    if (launched != rows) return MOE_ERR_CUDA;  // the two choices of kernel disagree (cannot happen)
  } else {
    st = launch_grouped_topk(gating, T, E, G, kg, topk, scoring, renorm, rsf, topk_weights, topk_ids, s, zero_rows,
                             zero_cols, nullptr, 0);
    if (st != MOE_OK) return st;
  }
  stage_mark(1, s);
  if (rows > 0)
    return launch_align_from_tile_hists(topk_ids, num_pairs, E, block_m, sorted_ids, expert_ids, offsets, ntpp,
                                        tile_hist, rows, tpr * topk, s, sorted_tok, topk, tile_counter);
  return launch_align(topk_ids, num_pairs, E, block_m, sorted_ids, expert_ids, offsets, ntpp, align_scratch, err, s,
                      sorted_tok, topk, tile_counter);
}

}  // namespace
}  // namespace moe

extern "C" void moe_set_stage_events(void* const* events, int n) {
  moe::g_num_stage_events = (events && n > 0) ? (n < 8 ? n : 8) : 0;
  for (int i = 0; i < moe::g_num_stage_events; ++i) moe::g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
}

extern "C" size_t moe_fused_forward_workspace_size(int T, int H, int I, int E, int topk) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0) return 0;
  // the layout of the kernel family that this problem size selects
  return moe::fused_layout(T, H, I, E, topk, moe::choose_plan(T, E, topk).block_m).total;
}

extern "C" moe_status_t moe_fused_forward(const void* x, const float* gating, const void* w_gate_up,
                                          const void* w_down, int T, int H, int I, int E, int num_expert_group,
                                          int topk_group, int topk, int scoring, int renormalize,
                                          float routed_scaling_factor, void* y, float* topk_weights,
                                          int32_t* topk_ids, void* ws, size_t ws_bytes, void* stream) {
  using namespace moe;
  moe_status_t st = validate_routing(T, E, num_expert_group, topk_group, topk, scoring);
  if (st != MOE_OK) return st;
  if (H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (!w_gate_up || !w_down) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !gating || !y || !topk_weights || !topk_ids)) return MOE_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(gating) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (static_cast<long long>(T) * topk >= (1ll << 30) || static_cast<long long>(T) * H >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED;
  const Plan plan = choose_plan(T, E, topk);
  const FusedLayout L = fused_layout(T, H, I, E, topk, plan.block_m);
  if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;

  cudaStream_t s = as_stream(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(w);
  int* tile_counter = err + 1;  // gate_up tile claims: zeroed by the align step
  int32_t* sorted_ids = reinterpret_cast<int32_t*>(w + L.sorted_ids);
  int32_t* sorted_tok = reinterpret_cast<int32_t*>(w + L.sorted_tok);
  int32_t* expert_ids = reinterpret_cast<int32_t*>(w + L.expert_ids);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.expert_offsets);
  int32_t* ntpp = reinterpret_cast<int32_t*>(w + L.ntpp);
  __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(w + L.h);
  float* y_acc = reinterpret_cast<float*>(w + L.y_acc);
  const int num_pairs = T * topk;

  // The fp32 accumulator of the down pass is cleared by the one-SM gate_up
  // kernel's epilogue warps while its first tiles run, else by the routing
  // kernel (each token's row).
  const bool gate_up_clears = !plan.swap;
  stage_mark(0, s);
  st = route_and_align(gating, T, E, num_expert_group, topk_group, topk, scoring, renormalize, routed_scaling_factor,
                       topk_weights, topk_ids, gate_up_clears ? nullptr : y_acc, H, plan.block_m, sorted_ids,
                       expert_ids, offsets, ntpp, w + L.align_scratch, err, sorted_tok, tile_counter, s);
  if (st != MOE_OK) return st;
  stage_mark(2, s);
  const size_t n4 = static_cast<size_t>(T) * H / 4;
  if (plan.swap)
    st = launch_swap_gate_up(static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_gate_up),
                             sorted_ids, offsets, h, err, num_pairs, topk, H, I, E, plan.nmax, s);
  else
    st = launch_gemm_gate_up_pairs(static_cast<const __nv_bfloat16*>(x),
                                   static_cast<const __nv_bfloat16*>(w_gate_up), sorted_tok, offsets, h, err,
                                   num_pairs, topk, H, I, E, y_acc, static_cast<size_t>(T) * H, tile_counter, s);
  if (st != MOE_OK) return st;
  stage_mark(3, s);
  if (plan.swap)
    st = launch_swap_down(h, static_cast<const __nv_bfloat16*>(w_down), sorted_ids, offsets, topk_weights, y_acc, err,
                          num_pairs, topk, L.cap, H, I, E, plan.nmax, s);
  else
    st = launch_gemm_down(h, static_cast<const __nv_bfloat16*>(w_down), sorted_ids, expert_ids, ntpp, topk_weights,
                          y_acc, err, num_pairs, topk, L.cap, H, I, E, s);
  if (st != MOE_OK) return st;
  stage_mark(4, s);
  st = launch_pdl(cast_f32_bf16_kernel, dim3(grid_for(n4)), dim3(256), 0, s,
                  reinterpret_cast<const float4*>(y_acc), reinterpret_cast<uint2*>(y), n4);
  if (st != MOE_OK) return st;
  stage_mark(5, s);
  return MOE_OK;
}

extern "C" size_t moe_fused_forward_fp8_workspace_size(int T, int H, int I, int E, int topk) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0) return 0;
  return moe::fp8_layout(T, H, I, E, topk).total;
}

extern "C" moe_status_t moe_fused_forward_fp8(const void* x, const float* gating, const void* w_gate_up,
                                              const float* scales_gate_up, const void* w_down,
                                              const float* scales_down, int T, int H, int I, int E,
                                              int num_expert_group, int topk_group, int topk, int scoring,
                                              int renormalize, float routed_scaling_factor, void* y,
                                              float* topk_weights, int32_t* topk_ids, void* ws, size_t ws_bytes,
                                              void* stream) {
  using namespace moe;
  moe_status_t st = validate_routing(T, E, num_expert_group, topk_group, topk, scoring);
  if (st != MOE_OK) return st;
  if (H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (!w_gate_up || !w_down || !scales_gate_up || !scales_down) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !gating || !y || !topk_weights || !topk_ids)) return MOE_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(gating) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(y) ||
      !aligned16(scales_gate_up) || !aligned16(scales_down))
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (static_cast<long long>(T) * topk >= (1ll << 30) || static_cast<long long>(T) * H >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED;
  const Fp8Layout L = fp8_layout(T, H, I, E, topk);
  if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;

  cudaStream_t s = as_stream(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(w);
  int* tile_counter = err + 1;  // gate_up tile claims: zeroed by the align step
  int32_t* sorted_ids = reinterpret_cast<int32_t*>(w + L.base.sorted_ids);
  int32_t* sorted_tok = reinterpret_cast<int32_t*>(w + L.base.sorted_tok);
  int32_t* expert_ids = reinterpret_cast<int32_t*>(w + L.base.expert_ids);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.base.expert_offsets);
  int32_t* ntpp = reinterpret_cast<int32_t*>(w + L.base.ntpp);
  __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(w + L.base.h);
  float* y_acc = reinterpret_cast<float*>(w + L.base.y_acc);
  uint8_t* qx = w + L.qx;
  float* sx = reinterpret_cast<float*>(w + L.sx);
  uint8_t* qh = w + L.qh;
  float* sh = reinterpret_cast<float*>(w + L.sh);
  const int num_pairs = T * topk;
  const int cap = L.base.cap;
  const Plan plan = choose_plan(T, E, topk);

  stage_mark(0, s);
  // x's per-token codes depend on x alone: quantised on the side stream while routing
  // and align run here, joined before gate_up reads them.
  SideStream* side = side_stream();
  if (side) {
    if (cudaEventRecord(side->fork, s) != cudaSuccess || cudaStreamWaitEvent(side->st, side->fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    st = launch_quant_rows_e4m3_bf16(static_cast<const __nv_bfloat16*>(x), T, H, qx, sx, nullptr, side->st);
    if (st != MOE_OK) return st;
    if (cudaEventRecord(side->join, side->st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // decode-sized problems: the swap-AB kernels, whose accumulator rows the routing kernel clears
  st = route_and_align(gating, T, E, num_expert_group, topk_group, topk, scoring, renormalize, routed_scaling_factor,
                       topk_weights, topk_ids, plan.swap ? y_acc : nullptr, H, plan.block_m, sorted_ids, expert_ids,
                       offsets, ntpp, w + L.base.align_scratch, err, sorted_tok, tile_counter, s);
  if (st != MOE_OK) return st;
  stage_mark(2, s);
  if (side) {
    if (cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    st = launch_quant_rows_e4m3_bf16(static_cast<const __nv_bfloat16*>(x), T, H, qx, sx, nullptr, s);
    if (st != MOE_OK) return st;
  }
  stage_mark(3, s);
  if (plan.swap)
    st = launch_swap_gate_up_fp8(qx, sx, static_cast<const uint8_t*>(w_gate_up), scales_gate_up, sorted_ids, offsets,
                                 h, err, num_pairs, topk, H, I, E, s);
  else
    st = launch_gemm_gate_up_pairs_fp8(qx, sx, static_cast<const uint8_t*>(w_gate_up), scales_gate_up, sorted_tok,
                                       offsets, h, err, H, I, E, y_acc, static_cast<size_t>(T) * H, tile_counter, s);
  if (st != MOE_OK) return st;
  stage_mark(4, s);
  st = launch_quant_rows_e4m3_bf16(h, cap, I, qh, sh, ntpp, s);
  if (st != MOE_OK) return st;
  stage_mark(5, s);
  if (plan.swap)
    st = launch_swap_down_fp8(qh, sh, static_cast<const uint8_t*>(w_down), scales_down, sorted_ids, offsets,
                              topk_weights, y_acc, err, num_pairs, topk, cap, H, I, E, s);
  else
    st = launch_gemm_down_fp8(qh, sh, static_cast<const uint8_t*>(w_down), scales_down, sorted_ids, expert_ids,
                              ntpp, topk_weights, y_acc, err, num_pairs, topk, cap, H, I, E, s);
  if (st != MOE_OK) return st;
  stage_mark(6, s);
  const size_t n4 = static_cast<size_t>(T) * H / 4;
  st = launch_pdl(cast_f32_bf16_kernel, dim3(grid_for(n4)), dim3(256), 0, s,
                  reinterpret_cast<const float4*>(y_acc), reinterpret_cast<uint2*>(y), n4);
  if (st != MOE_OK) return st;
  stage_mark(7, s);
  return MOE_OK;
}
