// moe_router_topk: the router projection logits = x @ W_g^T, then grouped top-k.
//
// Follows the mini-sglang MoE chapter, MoEMLP.forward: the gate is a replicated
// linear layer of H inputs and E outputs whose output is the gating input of
// select_experts; the GroupedTopK blog's gating_output (section 二) is that
// output. The logits are fp32: every product of a bf16 x value and an fp32 W_g
// value is formed by an fp32 FMA, in increasing k within a K range, and the K
// ranges' partial sums are added in range order, so the result is deterministic
// (the same bits on every call and every device).
//
// Work is tiny next to the layer (T*E*H multiply-adds) and at decode sizes is
// bound by reading W_g once, so the projection runs on the CUDA cores: a CTA
// computes a 64-token x 64-expert tile over a K range with 4 x 4 outputs per
// thread, staging 32-wide K slices of x (widened to fp32) and W_g through
// double-buffered shared memory. When the tiles alone would leave most SMs idle
// (few tokens), K is split across CTAs; their partial tiles go to the workspace
// and a second kernel adds them in range order. The grouped top-k kernels then
// read the logits back (from L2 at these sizes).
#include "common.cuh"

namespace moe {

moe_status_t validate_routing(int T, int E, int G, int kg, int k, int scoring);
moe_status_t launch_grouped_topk(const float* gating, int T, int E, int G, int kg, int k, int scoring, int renorm,
                                 float rsf, float* w, int32_t* ids, cudaStream_t s, float* zero_rows, int zero_cols,
                                 int* zero_cnt, int cnt_per_row);

namespace {

constexpr int kRT = 64;          // tokens per tile
constexpr int kRE = 64;          // experts per tile
constexpr int kRK = 32;          // K per staged slice
constexpr int kRPad = kRK + 4;   // shared row pitch (floats): 16-byte rows, conflict-free column reads
constexpr int kRThreads = 256;
constexpr int kRTargetCtas = 320;  // about two CTAs per SM on a 152-SM part
constexpr int kRMinSlices = 4;     // K slices per CTA at least, when K is split

// K ranges: every (tile, range) pair is one CTA. A pure function of the sizes, so
// the workspace size is known on the host without a device query.
int router_ksplit(int T, int H, int E) {
  const long long tiles = static_cast<long long>(cdiv(T, kRT)) * cdiv(E, kRE);
  const int nk = H / kRK;
  long long want = (kRTargetCtas + tiles - 1) / tiles;
  const int most = nk / kRMinSlices > 0 ? nk / kRMinSlices : 1;
  if (want > most) want = most;
  return want < 1 ? 1 : static_cast<int>(want);
}

// out[ks][t][e] (ks = blockIdx.z) = sum over the CTA's K slices of x[t, k] * wg[e, k].
__global__ void __launch_bounds__(kRThreads) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                                  const float* __restrict__ wg, int T, int H, int E,
                                                                  int ksplit, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) float xs[2][kRT][kRPad];
  __shared__ __align__(16) float wsm[2][kRE][kRPad];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.y * kRT;
  const int e0 = blockIdx.x * kRE;
  const int ks = blockIdx.z;
  const int nk = H / kRK;
  const int c0 = static_cast<int>(static_cast<long long>(ks) * nk / ksplit);
  const int c1 = static_cast<int>(static_cast<long long>(ks + 1) * nk / ksplit);

  // Loaders. x slice: 64 rows x 32 bf16 = 256 chunks of 8 bf16, one per thread.
  // W_g slice: 64 rows x 32 fp32 = 512 chunks of 4 floats, two per thread (rows r, r + 32).
  const int xr = tid >> 2, xc = (tid & 3) * 8;
  const int wr = tid >> 3, wc = (tid & 7) * 4;
  const bool xok = t0 + xr < T;
  const bool wok0 = e0 + wr < E, wok1 = e0 + wr + 32 < E;
  const __nv_bfloat16* xp = x + static_cast<size_t>(xok ? t0 + xr : 0) * H + xc;
  const float* wp0 = wg + static_cast<size_t>(wok0 ? e0 + wr : 0) * H + wc;
  const float* wp1 = wg + static_cast<size_t>(wok1 ? e0 + wr + 32 : 0) * H + wc;
  uint4 xv = make_uint4(0u, 0u, 0u, 0u);
  float4 wv0 = make_float4(0.f, 0.f, 0.f, 0.f), wv1 = wv0;
  auto load = [&](int c) {
    const int k = c * kRK;
    if (xok) xv = __ldg(reinterpret_cast<const uint4*>(xp + k));
    if (wok0) wv0 = __ldg(reinterpret_cast<const float4*>(wp0 + k));
    if (wok1) wv1 = __ldg(reinterpret_cast<const float4*>(wp1 + k));
  };
  auto store = [&](int buf) {
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
    const float2 a = __bfloat1622float2(h2[0]), b = __bfloat1622float2(h2[1]);
    const float2 c = __bfloat1622float2(h2[2]), d = __bfloat1622float2(h2[3]);
    *reinterpret_cast<float4*>(&xs[buf][xr][xc]) = make_float4(a.x, a.y, b.x, b.y);
    *reinterpret_cast<float4*>(&xs[buf][xr][xc + 4]) = make_float4(c.x, c.y, d.x, d.y);
    *reinterpret_cast<float4*>(&wsm[buf][wr][wc]) = wv0;
    *reinterpret_cast<float4*>(&wsm[buf][wr + 32][wc]) = wv1;
  };

  // Thread (ty, tx) owns tokens ty + 16 i and experts tx + 16 j (i, j < 4).
  const int ty = tid >> 4, tx = tid & 15;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  if (c0 < c1) {
    load(c0);
    store(0);
  }
  __syncthreads();
  for (int c = c0; c < c1; ++c) {
    const int buf = (c - c0) & 1;
    if (c + 1 < c1) load(c + 1);
#pragma unroll
    for (int kk = 0; kk < kRK; kk += 4) {
      float4 a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(&xs[buf][ty + 16 * i][kk]);
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = *reinterpret_cast<const float4*>(&wsm[buf][tx + 16 * j][kk]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float s = acc[i][j];
          s = fmaf(a[i].x, b[j].x, s);
          s = fmaf(a[i].y, b[j].y, s);
          s = fmaf(a[i].z, b[j].z, s);
          s = fmaf(a[i].w, b[j].w, s);
          acc[i][j] = s;
        }
    }
    if (c + 1 < c1) store(buf ^ 1);
    __syncthreads();
  }

  float* o = out + static_cast<size_t>(ks) * T * E;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty + 16 * i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx + 16 * j;
      if (e < E) o[static_cast<size_t>(t) * E + e] = acc[i][j];
    }
  }
}

// logits[i] = part[0][i] + part[1][i] + ... + part[ksplit - 1][i], in that order.
__global__ void __launch_bounds__(256) router_reduce_kernel(const float* __restrict__ part, size_t n, int ksplit,
                                                            float* __restrict__ logits) {
  pdl_trigger();
  pdl_wait();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n; i += stride) {
    float s = part[i];
    for (int k = 1; k < ksplit; ++k) s += part[static_cast<size_t>(k) * n + i];
    logits[i] = s;
  }
}

size_t router_ws_bytes(int T, int H, int E) {
  const int ks = router_ksplit(T, H, E);
  return ks > 1 ? align_up(static_cast<size_t>(ks) * T * E * sizeof(float), 256) : 0;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_router_topk_workspace_size(int T, int H, int E) {
  if (T < 0 || H <= 0 || E <= 0 || H % moe::kRK != 0) return 0;
  return moe::router_ws_bytes(T, H, E);
}

extern "C" moe_status_t moe_router_topk(const void* x, const float* w_gate, int T, int H, int E,
                                        int num_expert_group, int topk_group, int topk, int scoring, int renormalize,
                                        float routed_scaling_factor, float* router_logits, float* topk_weights,
                                        int32_t* topk_ids, void* ws, size_t ws_bytes, void* stream) {
  using namespace moe;
  moe_status_t st = validate_routing(T, E, num_expert_group, topk_group, topk, scoring);
  if (st != MOE_OK) return st;
  if (H <= 0 || !w_gate) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !router_logits || !topk_weights || !topk_ids)) return MOE_ERR_INVALID_ARG;
  if (H % kRK != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(router_logits)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (static_cast<long long>(T) * E >= (1ll << 31) || static_cast<long long>(T) * H >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED;
  const int ksplit = router_ksplit(T, H, E);
  const size_t need = router_ws_bytes(T, H, E);
  if (need > 0 && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0))
    return MOE_ERR_WORKSPACE;

  cudaStream_t s = as_stream(stream);
  float* part = ksplit > 1 ? static_cast<float*>(ws) : router_logits;
  const dim3 grid(cdiv(E, kRE), cdiv(T, kRT), ksplit);
  st = launch_pdl(router_logits_kernel, grid, dim3(kRThreads), 0, s, static_cast<const __nv_bfloat16*>(x), w_gate, T,
                  H, E, ksplit, part);
  if (st != MOE_OK) return st;
  if (ksplit > 1) {
    const size_t n = static_cast<size_t>(T) * E;
    const size_t want = (n + 255) / 256;
    const int sms = num_sms() > 0 ? num_sms() : 148;
    const int blocks = static_cast<int>(want < static_cast<size_t>(4 * sms) ? want : static_cast<size_t>(4 * sms));
    st = launch_pdl(router_reduce_kernel, dim3(blocks), dim3(256), 0, s, static_cast<const float*>(part), n, ksplit,
                    router_logits);
    if (st != MOE_OK) return st;
  }
  return launch_grouped_topk(router_logits, T, E, num_expert_group, topk_group, topk, scoring, renormalize,
                             routed_scaling_factor, topk_weights, topk_ids, s, nullptr, 0, nullptr, 0);
}
