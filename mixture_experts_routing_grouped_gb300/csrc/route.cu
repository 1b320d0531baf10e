// Grouped top-k routing: 8 lanes per token (the segmented kernel) where the shape
// allows it, else one warp per token; everything in registers.
//
// Follows "GroupedTopK 算子优化入门" section 三 (score, per-group max, top
// groups, mask, top-k, renormalise, scale) with the fusion plan of its
// section 六 (one program per token, only the k weights and k ids are written)
// and the simplification of section 七: both score functions are strictly
// increasing, so groups and experts are selected on the logits themselves and
// only the k selected logits are exponentiated when the weights renormalise.
//
// Segmented kernel (grouped_topk_seg_kernel): a token is L = 8 lanes of a warp,
// lane s holding experts [s*P, (s+1)*P) after the CTA's logits are staged in
// shared memory; its selection rounds are L-lane segment maxima plus a ballot.
// The warp-per-token kernels below serve the shapes it does not cover.
//
// Warp-per-token kernels: lane l holds the logits of experts [l*VPL, (l+1)*VPL). Warp-wide maxima and
// the lowest index among equal maxima come from redux.sync, so ties resolve to
// the lower expert (or group) index. The fast kernel (E = 32*VPL, power-of-two
// group count) reduces the float logits directly; the generic kernel (any E and
// G) reduces order-preserving unsigned keys of the logits.
#include "common.cuh"
#include "ptx.cuh"  // smem_u32

#include <cuda_runtime.h>
#include <math_constants.h>

namespace moe {

bool make_tmap_f32_32x32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);

namespace {

// Below this many tokens the segmented kernels (a single wave, no pipeline to fill) are faster.
constexpr int kTptMinTokens = 8192;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) == 0) b = 0;  // -0 and +0 compare equal
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Rows of the layer's fp32 accumulator (and per-row counters) that the routing
// warp of a token clears on the way out, so that the fused forward needs no
// separate clearing kernel. Null pointers: nothing to clear.
struct RouteZero {
  float4* rows;
  int row_f4;      // float4s per token row
  int* cnt;
  int cnt_per_row;
  int32_t* hist;   // segmented kernel: one row of E expert counts per CTA (null: none)
  int* err;        // device error word for ids the counts cannot take (null: none)
};

__device__ __forceinline__ void zero_token_rows(const RouteZero& z, int token, int lane) {
  if (z.rows) {
    float4* r = z.rows + static_cast<size_t>(token) * z.row_f4;
    for (int i = lane; i < z.row_f4; i += 32) r[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (z.cnt) {
    int* c = z.cnt + static_cast<size_t>(token) * z.cnt_per_row;
    for (int i = lane; i < z.cnt_per_row; i += 32) c[i] = 0;
  }
}

__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Weights of the k selections held by lanes 0..k-1 (blog 3.6 / section 七).
__device__ __forceinline__ float route_weight(float x, bool active, const float* v, int nv, int base, int E,
                                              int scoring, int renorm, float rsf) {
  float w;
  if (scoring == MOE_SCORE_SOFTMAX) {
    if (renorm) {
      // softmax over the selected logits only: the full denominator cancels
      const float x0 = __shfl_sync(0xffffffffu, x, 0);
      const float ex = active ? expf(x - x0) : 0.f;
      w = ex / warp_sum(ex);
    } else {
      float lmax = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < nv; ++j)
        if (base + j < E) lmax = fmaxf(lmax, v[j]);
      const float gmax = warp_max_f32(lmax);
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < nv; ++j)
        if (base + j < E) part += expf(v[j] - gmax);
      const float den = warp_sum(part);
      w = active ? expf(x - gmax) / den : 0.f;
    }
  } else {
    const float sg = active ? 1.0f / (1.0f + expf(-x)) : 0.f;
    w = renorm ? sg / warp_sum(sg) : sg;
  }
  return w * rsf;
}

// Fast path: E = 32 * VPL and G a power of two (a group spans 32 / G whole lanes).
// Group maxima come from segmented shuffles, group selection from each group's
// rank (no serial chain), and each lane caches its best two candidates so that
// only a lane that wins twice rescans its logits.
template <int VPL>
__global__ void __launch_bounds__(256) grouped_topk_fast_kernel(const float* __restrict__ gating, int T, int G,
                                                                int topk_group, int topk, int scoring, int renorm,
                                                                float rsf, float* __restrict__ out_w,
                                                                int32_t* __restrict__ out_ids, RouteZero zero) {
  pdl_trigger();
  pdl_wait();
  constexpr int E = 32 * VPL;
  const int token = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (token >= T) return;
  const float* row = gating + static_cast<size_t>(token) * E;
  const int base = lane * VPL;
  float v[VPL];
  if constexpr (VPL % 4 == 0) {
#pragma unroll
    for (int q = 0; q < VPL / 4; ++q) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + base) + q);
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < VPL; ++j) v[j] = __ldg(row + base + j);
  }

  // 3.2 / 3.3: group maximum over the group's lanes, then the group's rank.
  bool selected = true;
  if (G > 1) {
    const int lpg = 32 / G;
    float gk = v[0];
#pragma unroll
    for (int j = 1; j < VPL; ++j) gk = fmaxf(gk, v[j]);
    for (int o = 1; o < lpg; o <<= 1) gk = fmaxf(gk, __shfl_xor_sync(0xffffffffu, gk, o));
    const int my_g = lane / lpg;
    int rank = 0;
    for (int g = 0; g < G; ++g) {
      const float o = __shfl_sync(0xffffffffu, gk, g * lpg);
      rank += (o > gk || (o == gk && g < my_g)) ? 1 : 0;
    }
    selected = rank < topk_group;
  }

  // 3.4 / 3.5: the lane's best two candidates (ties keep the lower index).
  float best = -CUDART_INF_F, second = -CUDART_INF_F;
  int bidx = 0x7fffffff, sidx = 0x7fffffff;
  uint32_t taken = 0;
  if (selected) {
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      if (v[j] > best) { second = best; sidx = bidx; best = v[j]; bidx = base + j; }
      else if (v[j] > second) { second = v[j]; sidx = base + j; }
    }
  }
  bool second_valid = true;
  float my_x = 0.f;
  int my_id = 0;
  for (int it = 0; it < topk; ++it) {
    const float m = warp_max_f32(best);
    const uint32_t w = __reduce_min_sync(0xffffffffu, best == m ? static_cast<uint32_t>(bidx) : 0x7fffffffu);
    if (lane == it) { my_x = m; my_id = static_cast<int>(w); }
    if (bidx == static_cast<int>(w) && w != 0x7fffffffu) {
      taken |= 1u << (bidx - base);
      if (second_valid) {
        best = second; bidx = sidx;
        second_valid = false;
      } else {
        best = -CUDART_INF_F; bidx = 0x7fffffff;
        second = -CUDART_INF_F; sidx = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          if ((taken >> j) & 1u) continue;
          if (v[j] > best) { second = best; sidx = bidx; best = v[j]; bidx = base + j; }
          else if (v[j] > second) { second = v[j]; sidx = base + j; }
        }
        second_valid = true;
      }
    }
  }

  const bool active = lane < topk;
  const float wgt = route_weight(my_x, active, v, VPL, base, E, scoring, renorm, rsf);
  if (active) {
    out_w[static_cast<size_t>(token) * topk + lane] = wgt;
    out_ids[static_cast<size_t>(token) * topk + lane] = my_id;
  }
  zero_token_rows(zero, token, lane);
}

template <int VPL>
__global__ void __launch_bounds__(256) grouped_topk_kernel(const float* __restrict__ gating, int T, int E, int G,
                                                           int topk_group, int topk, int scoring, int renorm,
                                                           float rsf, float* __restrict__ out_w,
                                                           int32_t* __restrict__ out_ids, RouteZero zero) {
  pdl_trigger();
  pdl_wait();
  const int token = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (token >= T) return;
  const float* row = gating + static_cast<size_t>(token) * E;
  const int base = lane * VPL;
  const int P = E / G;

  float v[VPL];
  if constexpr (VPL % 4 == 0) {
    if ((E & 3) == 0) {
#pragma unroll
      for (int q = 0; q < VPL / 4; ++q) {
        if (base + 4 * q < E) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(row + base + 4 * q));
          v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
        } else {
          v[4 * q] = v[4 * q + 1] = v[4 * q + 2] = v[4 * q + 3] = 0.f;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < VPL; ++j) v[j] = (base + j < E) ? __ldg(row + base + j) : 0.f;
    }
  } else {
#pragma unroll
    for (int j = 0; j < VPL; ++j) v[j] = (base + j < E) ? __ldg(row + base + j) : 0.f;
  }

  uint32_t key[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) key[j] = (base + j < E) ? order_key(v[j]) : 0u;
  int grp[VPL];  // group of each of the lane's experts, without a division per element
  {
    int g = base / P, next = (base / P + 1) * P;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      if (base + j >= next) { ++g; next += P; }
      grp[j] = g;
    }
  }

  // 3.2: group maxima. Lane g (< G) ends up holding the key of group g.
  uint32_t my_gkey = 0;
  if (P % VPL == 0) {
    // every lane's experts lie in one group
    uint32_t lmax = 0;
#pragma unroll
    for (int j = 0; j < VPL; ++j) lmax = max(lmax, key[j]);
    const int my_group = base / P;
    for (int g = 0; g < G; ++g) {
      const uint32_t m = __reduce_max_sync(0xffffffffu, my_group == g ? lmax : 0u);
      if (lane == g) my_gkey = m;
    }
  } else {
    for (int g = 0; g < G; ++g) {
      uint32_t lmax = 0;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (grp[j] == g) lmax = max(lmax, key[j]);
      const uint32_t m = __reduce_max_sync(0xffffffffu, lmax);
      if (lane == g) my_gkey = m;
    }
  }

  // 3.3: top `topk_group` groups (ties -> lower group index).
  uint32_t sel_groups = 0;  // bit g set <=> group g kept (G <= 32)
  {
    uint32_t cand = (lane < G) ? my_gkey : 0u;
    bool taken = false;
    for (int it = 0; it < topk_group; ++it) {
      const uint32_t m = __reduce_max_sync(0xffffffffu, taken ? 0u : cand);
      const uint32_t w = __reduce_min_sync(0xffffffffu, (!taken && lane < G && cand == m) ? lane : 64u);
      sel_groups |= 1u << w;
      if (lane == static_cast<int>(w)) taken = true;
    }
  }

  // 3.4: mask experts of unselected groups (key 0 is below every finite logit).
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    if (base + j < E && !((sel_groups >> grp[j]) & 1u)) key[j] = 0u;
  }

  // 3.5: top `topk` experts (ties -> lower expert index).
  uint32_t lbest = 0;
  int lidx = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < VPL; ++j)
    if (key[j] > lbest) { lbest = key[j]; lidx = base + j; }
  uint32_t my_key = 0;  // lane `it` keeps the it-th selection
  int my_id = 0;
  for (int it = 0; it < topk; ++it) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, lbest);
    const uint32_t w = __reduce_min_sync(0xffffffffu, lbest == m ? static_cast<uint32_t>(lidx) : 0x7fffffffu);
    if (lane == it) { my_key = m; my_id = static_cast<int>(w); }
    if (lidx == static_cast<int>(w)) {  // owner removes the winner, finds its next best
      lbest = 0; lidx = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        if (base + j == static_cast<int>(w)) key[j] = 0u;
        if (key[j] > lbest) { lbest = key[j]; lidx = base + j; }
      }
    }
  }

  // 3.6: weights.
  const bool active = lane < topk;
  const float x = active ? key_to_float(my_key) : 0.f;
  float w;
  if (scoring == MOE_SCORE_SOFTMAX) {
    if (renorm) {
      // softmax over the selected logits only: the full denominator cancels (section 七)
      const float x0 = __shfl_sync(0xffffffffu, x, 0);
      const float ex = active ? expf(x - x0) : 0.f;
      const float s = warp_sum(ex);
      w = ex / s;
    } else {
      uint32_t lmax = 0;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (base + j < E) lmax = max(lmax, order_key(v[j]));
      const float gmax = key_to_float(__reduce_max_sync(0xffffffffu, lmax));
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (base + j < E) part += expf(v[j] - gmax);
      const float den = warp_sum(part);
      w = active ? expf(x - gmax) / den : 0.f;
    }
  } else {
    const float s = active ? 1.0f / (1.0f + expf(-x)) : 0.f;
    w = s;
    if (renorm) w = s / warp_sum(s);
  }
  w *= rsf;
  if (active) {
    out_w[static_cast<size_t>(token) * topk + lane] = w;
    out_ids[static_cast<size_t>(token) * topk + lane] = my_id;
  }
  zero_token_rows(zero, token, lane);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Segmented kernel: L lanes per token (32 / L tokens per warp, 256 / L per CTA),
// lane s of a token holding experts [s*P, (s+1)*P), and every real group of E/G
// experts spanning L/G whole lanes. With one token per warp the k selection
// rounds and the group ranking dominated the instruction count; here they are
// L-lane segment reductions shared by 32 / L tokens.
//
// The CTA's logits (256 rows of P floats, one row per lane) are loaded with
// coalesced 16-byte loads and stored to shared memory with the 16-byte chunk
// bits of each address XORed with the address bits above the 128-byte line, so
// that lanes reading chunk j of consecutive rows hit distinct banks. (Loading
// each lane's own row directly touches 32 lines per warp instruction.)
//
// Phase 1 (3.2 / 3.3): row maxima, group maxima over the group's lanes, each
// group's rank among the token's G groups. Phase 2 (3.4 / 3.5): the rows of the
// selected groups are re-read from shared memory, F = G / topk_group lanes per
// selected row and P / F values per lane, in increasing expert order across the
// segment, so that every lane works on candidates; each lane caches its best two
// (ties keep the lower expert index) and in each of the k rounds the segment
// maximum and its lowest lane (ballot) give the next expert. A lane caches its
// best four candidates (ties keep the lower expert index); only a lane that
// wins a fifth time looks for its next candidate, in one pass for the best
// value ranked below the one it just gave up. (Rebuilding a two-deep cache on a
// third win was most of the instructions.) K > 0 fixes topk at compile time so
// that the rounds unroll (K = 0: topk at run time).
constexpr int kSegThreads = 128;  // a CTA holds 128 lane-rows: 128 / L tokens

template <int P, int L, int F, int K>
__global__ void __launch_bounds__(kSegThreads, 6) grouped_topk_seg_kernel(const float* __restrict__ gating, int T,
                                                                          int G, int topk_group, int topk,
                                                                          int scoring, int renorm, float rsf,
                                                                          float* __restrict__ out_w,
                                                                          int32_t* __restrict__ out_ids,
                                                                          RouteZero zero) {
  pdl_trigger();
  pdl_wait();
  constexpr int kRowBytes = P * 4;
  constexpr int kChunks = P / 4;  // 16-byte chunks per row, = chunks loaded per thread
  constexpr int V = P / F;        // phase-2 values per lane
  constexpr uint32_t kSwzMask = kRowBytes >= 32 ? kRowBytes / 16 - 1 : 0;
  if (K > 0) topk = K;
  __shared__ __align__(1024) uint8_t rows[kSegThreads * kRowBytes];
  __shared__ int hist_s[P * L];
  const int tid = threadIdx.x;
  const uint32_t base = ptx::smem_u32(rows);
  auto chunk_addr = [&](int row, int j) {  // shared address of 16-byte chunk j of lane-row `row`
    uint32_t addr = static_cast<uint32_t>(row) * kRowBytes + j * 16;
    return base + (addr ^ (((addr >> 7) & kSwzMask) << 4));
  };
  {
    constexpr int E = P * L;
    const size_t n4 = static_cast<size_t>(T) * E / 4;
    const size_t first = static_cast<size_t>(blockIdx.x) * kSegThreads * kChunks;
    const float4* src = reinterpret_cast<const float4*>(gating) + first;
    float4 f[kChunks];
#pragma unroll
    for (int q = 0; q < kChunks; ++q) {
      const int c = tid + kSegThreads * q;
      f[q] = first + c < n4 ? __ldg(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < kChunks; ++q) {
      const int c = tid + kSegThreads * q;
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(chunk_addr(c / kChunks, c % kChunks)),
                   "f"(f[q].x), "f"(f[q].y), "f"(f[q].z), "f"(f[q].w)
                   : "memory");
    }
  }
  __syncthreads();

  const int lane = tid & 31;
  const int s = lane & (L - 1);
  const int seg0 = lane & ~(L - 1);
  const int trow0 = tid - s;  // lane-row of the token's first lane in the CTA
  const int token = static_cast<int>(blockIdx.x) * (kSegThreads / L) + tid / L;

  // Phase 1: own row's maximum, group maximum, group rank.
  float lm = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    float4 f;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                 : "r"(chunk_addr(tid, j))
                 : "memory");
    lm = max3f(lm, max3f(f.x, f.y, f.z), f.w);
  }
  const int lpg = L / G;
  float gm = lm;
  for (int o = 1; o < lpg; o <<= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
  bool selected = true;
  if (topk_group < G) {
    const int my_g = s / lpg;
    int rank = 0;
    for (int g = 0; g < G; ++g) {
      const float o = __shfl_sync(0xffffffffu, gm, seg0 + g * lpg);
      rank += (o > gm || (o == gm && g < my_g)) ? 1 : 0;
    }
    selected = rank < topk_group;
  }
  // Phase 2: lane s takes part s % F of the (s / F)-th selected row, in row order.
  const uint32_t rowmask = (__ballot_sync(0xffffffffu, selected) >> seg0) & (L == 32 ? 0xffffffffu : ((1u << L) - 1u));
  int my_row = s;
  if (F > 1) {
    uint32_t m = rowmask;
    for (int i = 0; i < s / F; ++i) m &= m - 1;  // drop the lowest selected rows before ours
    my_row = __ffs(m) - 1;
  }
  const bool has_row = F > 1 || selected;
  const int part = s % F;
  const int base_e = my_row * P + part * V;
  float v[V];
#pragma unroll
  for (int j = 0; j < V / 4; ++j) {
    float4 f;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                 : "r"(chunk_addr(trow0 + my_row, part * (V / 4) + j))
                 : "memory");
    v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
  }
  // best four of the lane's candidates (b1 >= b2 >= b3 >= b4); indices ascend
  // with j, so strict comparisons keep the lower index among equal values
  float b1 = -CUDART_INF_F, b2 = -CUDART_INF_F, b3 = -CUDART_INF_F, b4 = -CUDART_INF_F;
  int i1 = 0x7fffffff, i2 = 0x7fffffff, i3 = 0x7fffffff, i4 = 0x7fffffff;
  if (has_row) {
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const float x = v[j];
      const int ix = base_e + j;
      const bool p1 = x > b1, p2 = x > b2, p3 = x > b3, p4 = x > b4;
      b4 = p3 ? b3 : (p4 ? x : b4);
      i4 = p3 ? i3 : (p4 ? ix : i4);
      b3 = p2 ? b2 : (p3 ? x : b3);
      i3 = p2 ? i2 : (p3 ? ix : i3);
      b2 = p1 ? b1 : (p2 ? x : b2);
      i2 = p1 ? i1 : (p2 ? ix : i2);
      b1 = p1 ? x : b1;
      i1 = p1 ? ix : i1;
    }
  }
  float my_x = 0.f;
  int my_id = 0;
  const uint32_t segmask = L == 32 ? 0xffffffffu : (((1u << L) - 1u) << seg0);
#pragma unroll(K > 0 ? K : 1)
  for (int it = 0; it < topk; ++it) {
    float m = b1;
#pragma unroll
    for (int o = 1; o < L; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const uint32_t wm = __ballot_sync(0xffffffffu, b1 == m) & segmask;
    const int wl = __ffs(wm) - 1;
    const int wid = __shfl_sync(0xffffffffu, i1, wl & 31);
    if (s == it) { my_x = m; my_id = wid; }
    if (lane == wl) {
      const float lv = b1;
      const int li = i1;
      b1 = b2; i1 = i2;
      b2 = b3; i2 = i3;
      b3 = b4; i3 = i4;
      b4 = -CUDART_INF_F; i4 = 0x7fffffff;
      if (b1 == -CUDART_INF_F) {
        // cache exhausted: the best value ranked below (lv, li)
#pragma unroll
        for (int j = 0; j < V; ++j) {
          const bool below = v[j] < lv || (v[j] == lv && base_e + j > li);
          if (below && v[j] > b1) { b1 = v[j]; i1 = base_e + j; }
        }
      }
    }
  }

  // 3.6: weights of the topk selections held by segment lanes 0..topk-1.
  const bool active = s < topk;
  float w;
  if (scoring == MOE_SCORE_SOFTMAX) {
    if (renorm) {
      // softmax over the selected logits only: the full denominator cancels
      const float x0 = __shfl_sync(0xffffffffu, my_x, seg0);
      const float ex = active ? expf(my_x - x0) : 0.f;
      float sum = ex;
#pragma unroll
      for (int o = 1; o < L; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      w = ex / sum;
    } else {
      float tm = lm;
#pragma unroll
      for (int o = 1; o < L; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
      float part_sum = 0.f;
#pragma unroll
      for (int j = 0; j < kChunks; ++j) {
        float4 f;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                     : "r"(chunk_addr(tid, j))
                     : "memory");
        part_sum += expf(f.x - tm) + expf(f.y - tm) + expf(f.z - tm) + expf(f.w - tm);
      }
#pragma unroll
      for (int o = 1; o < L; o <<= 1) part_sum += __shfl_xor_sync(0xffffffffu, part_sum, o);
      w = active ? expf(my_x - tm) / part_sum : 0.f;
    }
  } else {
    const float sg = active ? 1.0f / (1.0f + expf(-my_x)) : 0.f;
    w = sg;
    if (renorm) {
      float sum = sg;
#pragma unroll
      for (int o = 1; o < L; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      w = sg / sum;
    }
  }
  w *= rsf;
  if (token < T) {
    if (active) {
      out_w[static_cast<size_t>(token) * topk + s] = w;
      out_ids[static_cast<size_t>(token) * topk + s] = my_id;
    }
    if (zero.rows) {
      float4* r = zero.rows + static_cast<size_t>(token) * zero.row_f4;
      for (int i = s; i < zero.row_f4; i += L) r[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (zero.cnt) {
      int* c = zero.cnt + static_cast<size_t>(token) * zero.cnt_per_row;
      for (int i = s; i < zero.cnt_per_row; i += L) c[i] = 0;
    }
  }
  // the CTA's expert counts (align's first pass over its tokens' pairs), when asked for
  if (zero.hist) {
    constexpr int E = P * L;
    for (int e = tid; e < E; e += kSegThreads) hist_s[e] = 0;
    __syncthreads();
    if (token < T && active) {
      if (static_cast<unsigned>(my_id) < static_cast<unsigned>(E)) atomicAdd(&hist_s[my_id], 1);
      else report_error(zero.err, MOE_DEVERR_EXPERT_ID);
    }
    __syncthreads();
    int32_t* row_out = zero.hist + static_cast<size_t>(blockIdx.x) * E;
    for (int e = tid; e < E; e += kSegThreads) row_out[e] = hist_s[e];
  }
}

// ----------------------------------------------------------------------------
// Thread-per-token kernel for the common shapes (E = 128 or 256, whole 8-expert
// units per group, topk = 8), fed by TMA.
//
// A persistent CTA per SM: one producer thread streams tiles of 32 tokens (their
// [32, E] fp32 logits) into shared-memory stages with 2D tensor loads (boxes of 32
// logits x 32 tokens, 128-byte swizzle, so that lane r reading its own row touches
// eight distinct bank groups per quarter-warp), and seven compute warps take the
// tiles in turn, lane r of a warp selecting for token r of its tile; each warp owns
// its own stages. The loads of the next tiles are in flight while the current ones
// are selected. The selection's dependent chains bound the kernel, so the stages are
// as many as shared memory holds (224 KB), for as many compute warps.
//
// Per token (GroupedTopK blog 3.2-3.6, on the logits as in its section 七):
//  1. maxima of every unit of 8 consecutive experts, and the group maxima from them;
//  2. the group ranks (greater maximum first, equal maxima to the lower group), and
//     the mask of the topk_group best groups;
//  3. a lower bound tau of the topk-th largest candidate: the topk-th largest of the
//     selected groups' unit maxima (distinct candidates, so at least topk are >= tau);
//  4. the candidates >= tau (about topk + 2 on Gaussian logits) are marked in bit
//     masks of the selected groups;
//  5. the marked candidates, in increasing index, are inserted into a sorted register
//     list of topk (value, index) pairs, strict comparisons keeping the lower index
//     first among equal values (rows with many equal values near the top just mark
//     more candidates).
// The weights follow as in the other kernels.
namespace tpt {

constexpr int kTile = 32;
constexpr int kComputeWarps = 7;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kK = 8;

template <int E>
struct Shape {
  static constexpr int kBoxes = E / 32;                 // 128-byte column boxes per row
  static constexpr int kUnits = E / 8;
  static constexpr int kStageBytes = kTile * E * 4;     // 32 KB at E = 256
  // each compute warp owns kDepth stages (one consumer per stage: its barriers are waited on in
  // order by one warp, so no wait can match an older phase of the same parity)
  static constexpr int kDepth = (224 * 1024) / kStageBytes / kComputeWarps > 0
                                    ? (224 * 1024) / kStageBytes / kComputeWarps : 1;
  static constexpr int kStages = kComputeWarps * kDepth;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kSmem = kBarOff + 2 * kStages * 8 + 16 + 1024;  // + alignment slack
  static_assert(kSmem <= 232448, "routing stages exceed the per-CTA shared memory");
  static_assert(E * 4 <= kStageBytes, "a tile's expert counts fit in its stage");
};

// Shared address of logit e of lane-row r in a stage (see the swizzle above).
template <int E>
__device__ __forceinline__ uint32_t logit_addr(uint32_t stage, int r, int e) {
  const int box = e >> 5, chunk = (e >> 2) & 7, word = e & 3;
  return stage + box * 4096 + r * 128 + (((chunk ^ (r & 7)) << 4) | (word << 2));
}

__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds_f32x4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}

// (x, ix) into the descending list (v, id) of kK entries; candidates arrive in
// increasing index, so a strict comparison puts x after every equal value.
__device__ __forceinline__ void insert_sorted(float (&v)[kK], int (&id)[kK], float x, int ix) {
  bool c[kK];
#pragma unroll
  for (int i = 0; i < kK; ++i) c[i] = x > v[i];
#pragma unroll
  for (int i = kK - 1; i > 0; --i) {
    const float vm = c[i - 1] ? v[i - 1] : x;
    const int im = c[i - 1] ? id[i - 1] : ix;
    v[i] = c[i] ? vm : v[i];
    id[i] = c[i] ? im : id[i];
  }
  v[0] = c[0] ? x : v[0];
  id[0] = c[0] ? ix : id[0];
}

template <int E, int G, int KG>
__global__ void __launch_bounds__(kThreads, 1) grouped_topk_tpt_kernel(const __grid_constant__ CUtensorMap map,
                                                                      int T, int ntiles, int scoring, int renorm,
                                                                      float rsf, float* __restrict__ out_w,
                                                                      int32_t* __restrict__ out_ids, int* err,
                                                                      int32_t* __restrict__ tile_hist) {
  pdl_trigger();
  pdl_wait();
  using S = Shape<E>;
  constexpr int P = E / G;              // experts per group
  constexpr int UPG = P / 8;            // units per group
  static_assert(P % 8 == 0, "groups of whole 8-expert units");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar_full = sbase + S::kBarOff;
  const uint32_t bar_empty = bar_full + S::kStages * 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kBarOff + 2 * S::kStages * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kStages; ++i) {
      ptx::mbar_init(bar_full + 8 * i, 1);
      ptx::mbar_init(bar_empty + 8 * i, 1);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // producer
    if (lane == 0) {
      ptx::prefetch_tmap(&map);
      // CTA-local tile i goes to warp i % W, its l = i / W -th tile, stage (i % W) * D + l % D
      auto stage_of = [](int i) { return (i % kComputeWarps) * S::kDepth + (i / kComputeWarps) % S::kDepth; };
      auto use_of = [](int i) { return (i / kComputeWarps) / S::kDepth; };  // earlier uses of that stage
      int issued = 0;
      for (int i = 0;; ++i) {
        const int tile = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
        if (tile >= ntiles) break;
        const int s = stage_of(i);
        if (use_of(i) > 0 && !ptx::mbar_wait(bar_empty + 8 * s, (use_of(i) - 1) & 1, abort_flag)) break;
        ptx::mbar_arrive_expect_tx(bar_full + 8 * s, S::kStageBytes);
        const uint32_t dst = sbase + s * S::kStageBytes;
#pragma unroll
        for (int b = 0; b < S::kBoxes; ++b) ptx::tma_load_2d(dst + b * 4096, &map, bar_full + 8 * s, b * 32, tile * kTile);
        issued = i + 1;
      }
      // every issued copy has landed before the CTA may exit (a no-op unless a wait gave up);
      // the last kStages tiles issued cover each stage once
      for (int j = issued - S::kStages > 0 ? issued - S::kStages : 0; j < issued; ++j)
        ptx::mbar_wait_drain(bar_full + 8 * stage_of(j), use_of(j) & 1);
    }
    return;
  }

  for (int l = 0;; ++l) {
    const int i = l * kComputeWarps + warp;
    const int tile = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    if (tile >= ntiles) break;
    const int s = warp * S::kDepth + l % S::kDepth;
    // the warp leaves as one (warp-wide shuffles and syncs follow)
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_full + 8 * s, (l / S::kDepth) & 1, abort_flag))) {
      if (lane == 0) report_error(err, MOE_DEVERR_TIMEOUT);
      break;
    }
    const uint32_t stage = sbase + s * S::kStageBytes;
    const int r = lane;

    // 1. unit and group maxima
    float um[S::kUnits];
#pragma unroll
    for (int b = 0; b < S::kBoxes; ++b) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 a = lds_f32x4(stage + b * 4096 + r * 128 + (((2 * u) ^ (r & 7)) << 4));
        const float4 c = lds_f32x4(stage + b * 4096 + r * 128 + (((2 * u + 1) ^ (r & 7)) << 4));
        um[b * 4 + u] = fmaxf(max3f(max3f(a.x, a.y, a.z), max3f(a.w, c.x, c.y), c.z), c.w);
      }
    }
    float gm[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float m = um[g * UPG];
#pragma unroll
      for (int u = 1; u < UPG; ++u) m = fmaxf(m, um[g * UPG + u]);
      gm[g] = m;
    }
    // 2. group ranks
    uint32_t sel = (G == 32) ? 0xffffffffu : ((1u << G) - 1u);
    if (KG < G) {
      int rank[G];
#pragma unroll
      for (int g = 0; g < G; ++g) rank[g] = 0;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int h = g + 1; h < G; ++h) {
          const bool h_first = gm[h] > gm[g];  // equal maxima: the lower group g goes first
          rank[g] += h_first ? 1 : 0;
          rank[h] += h_first ? 0 : 1;
        }
      sel = 0;
#pragma unroll
      for (int g = 0; g < G; ++g) sel |= (rank[g] < KG ? 1u : 0u) << g;
    }
    // 3. tau: the topk-th largest unit maximum among the selected groups' units (each unit
    //    maximum is a distinct candidate, so at least topk candidates are >= tau)
    float tau = -CUDART_INF_F;
    if (KG * UPG >= kK) {
      float t[kK];
#pragma unroll
      for (int q = 0; q < kK; ++q) t[q] = -CUDART_INF_F;
#pragma unroll
      for (int u = 0; u < S::kUnits; ++u) {
        const float x = ((sel >> (u / UPG)) & 1u) ? um[u] : -CUDART_INF_F;
#pragma unroll
        for (int q = kK - 1; q > 0; --q) t[q] = fmaxf(t[q], fminf(t[q - 1], x));
        t[0] = fmaxf(t[0], x);
      }
      tau = t[kK - 1];
    }
    // 4-5. per selected group (in increasing group order): a bit mask of its candidates >= tau,
    //      then the marked candidates inserted in increasing index into the sorted top-k
    float v[kK];
    int id[kK];
#pragma unroll
    for (int q = 0; q < kK; ++q) { v[q] = -CUDART_INF_F; id[q] = 0x7fffffff; }
    for (uint32_t rem = sel; rem; rem &= rem - 1) {
      const int g = __ffs(rem) - 1;
#pragma unroll 1
      for (int w = 0; w < (P + 31) / 32; ++w) {
        const int base = g * P + 32 * w;
        uint32_t m = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (32 * w + 4 * c >= P) break;
          const int e0 = base + 4 * c;
          const float4 f = lds_f32x4(stage + (e0 >> 5) * 4096 + r * 128 + ((((e0 >> 2) & 7) ^ (r & 7)) << 4));
          m |= ((f.x >= tau ? 1u : 0u) | (f.y >= tau ? 2u : 0u) | (f.z >= tau ? 4u : 0u) | (f.w >= tau ? 8u : 0u))
               << (4 * c);
        }
        while (m) {
          const int e = base + __ffs(m) - 1;
          m &= m - 1;
          insert_sorted(v, id, lds_f32(logit_addr<E>(stage, r, e)), e);
        }
      }
    }
    // softmax without renormalisation needs the full denominator: read the row once more and
    // add its E terms pairwise (depth log2(E): every term is positive, so the sum's relative
    // error stays within that many roundings)
    float den = 0.f, rmax = 0.f;
    if (scoring == MOE_SCORE_SOFTMAX && !renorm) {
      rmax = gm[0];
#pragma unroll
      for (int g = 1; g < G; ++g) rmax = fmaxf(rmax, gm[g]);
      float bs[S::kBoxes];
#pragma unroll
      for (int b = 0; b < S::kBoxes; ++b) {
        float cs[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 f = lds_f32x4(stage + b * 4096 + r * 128 + ((c ^ (r & 7)) << 4));
          cs[c] = (expf(f.x - rmax) + expf(f.y - rmax)) + (expf(f.z - rmax) + expf(f.w - rmax));
        }
        bs[b] = ((cs[0] + cs[1]) + (cs[2] + cs[3])) + ((cs[4] + cs[5]) + (cs[6] + cs[7]));
      }
#pragma unroll
      for (int h = S::kBoxes / 2; h >= 1; h /= 2)
#pragma unroll
        for (int b = 0; b < h; ++b) bs[b] += bs[b + h];
      den = bs[0];
    }
    __syncwarp();
    // the stage is free once read, unless the tile's expert counts are taken in it below
    if (!tile_hist && lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);

    // 3.6: weights (one reciprocal of the sum; each sigmoid as the correctly rounded 1 / (1 + e^-x))
    float w[kK];
    if (scoring == MOE_SCORE_SOFTMAX) {
      if (renorm) {
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < kK; ++q) { w[q] = expf(v[q] - v[0]); sum += w[q]; }
        const float inv = 1.0f / sum;
#pragma unroll
        for (int q = 0; q < kK; ++q) w[q] *= inv;
      } else {
        const float inv = 1.0f / den;
#pragma unroll
        for (int q = 0; q < kK; ++q) w[q] = expf(v[q] - rmax) * inv;
      }
    } else {
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < kK; ++q) { w[q] = __frcp_rn(1.0f + expf(-v[q])); sum += w[q]; }
      if (renorm) {
        const float inv = 1.0f / sum;
#pragma unroll
        for (int q = 0; q < kK; ++q) w[q] *= inv;
      }
    }
    const int token = tile * kTile + r;
    if (token < T) {
      float4* wp = reinterpret_cast<float4*>(out_w + static_cast<size_t>(token) * kK);
      int4* ip = reinterpret_cast<int4*>(out_ids + static_cast<size_t>(token) * kK);
      wp[0] = make_float4(w[0] * rsf, w[1] * rsf, w[2] * rsf, w[3] * rsf);
      wp[1] = make_float4(w[4] * rsf, w[5] * rsf, w[6] * rsf, w[7] * rsf);
      ip[0] = make_int4(id[0], id[1], id[2], id[3]);
      ip[1] = make_int4(id[4], id[5], id[6], id[7]);
    }
    // the tile's expert counts (align's first pass over these pairs), when asked for,
    // counted in the warp's own stage (its logits are no longer read), which is then freed
    if (tile_hist) {
      int* wh = reinterpret_cast<int*>(smem + s * S::kStageBytes);
      for (int e = lane; e < E; e += 32) wh[e] = 0;
      __syncwarp();
      if (token < T) {
#pragma unroll
        for (int q = 0; q < kK; ++q) {
          if (static_cast<unsigned>(id[q]) < static_cast<unsigned>(E)) atomicAdd(&wh[id[q]], 1);
          else report_error(err, MOE_DEVERR_EXPERT_ID);
        }
      }
      __syncwarp();
      int32_t* row_out = tile_hist + static_cast<size_t>(tile) * E;
      for (int e = lane; e < E; e += 32) row_out[e] = wh[e];
      // the next tile's copy into this stage (async proxy) follows these shared-memory writes
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
    }
  }
}

}  // namespace tpt

// Lanes per token for the segmented kernel (8, 16 or 32), or 0 when it does not
// apply: P = E / L must be 4, 8, 16 or 32, every group must span whole lanes
// (G divides L) and the topk results must fit one per lane (topk <= L).
int seg_lanes(int E, int G, int k) {
  for (int L = 8; L <= 32; L <<= 1) {
    if (E % L != 0) continue;
    const int P = E / L;
    if ((P != 4 && P != 8 && P != 16 && P != 32) || L % G != 0 || k > L) continue;
    return L;
  }
  return 0;
}

template <int P, int L, int F>
moe_status_t launch_seg_f(const float* gating, int T, int G, int kg, int k, int scoring, int renorm, float rsf,
                          float* w, int32_t* ids, const RouteZero& z, cudaStream_t s) {
  const int grid = cdiv(T, kSegThreads / L);
  if (k == 8 && L >= 8)
    return launch_pdl(grouped_topk_seg_kernel<P, L, F, 8>, dim3(grid), dim3(kSegThreads), 0, s, gating, T, G, kg, k,
                      scoring, renorm, rsf, w, ids, z);
  return launch_pdl(grouped_topk_seg_kernel<P, L, F, 0>, dim3(grid), dim3(kSegThreads), 0, s, gating, T, G, kg, k,
                    scoring, renorm, rsf, w, ids, z);
}

template <int P, int L>
moe_status_t launch_seg(const float* gating, int T, int G, int kg, int k, int scoring, int renorm, float rsf,
                        float* w, int32_t* ids, const RouteZero& z, cudaStream_t s) {
  // F = G / topk_group lanes share a selected row in phase 2 (1 when that is not
  // 2 or 4, or leaves fewer than 4 values per lane)
  const int F = (G % kg == 0) ? G / kg : 1;
  if (F == 2 && P >= 8) return launch_seg_f<P, L, 2>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  if (F == 4 && P >= 16) return launch_seg_f<P, L, 4>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  return launch_seg_f<P, L, 1>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
}

template <int VPL>
moe_status_t launch_fast(const float* gating, int T, int G, int kg, int k, int scoring, int renorm, float rsf,
                         float* w, int32_t* ids, const RouteZero& z, cudaStream_t s) {
  const int threads = 256;
  const int blocks = cdiv(T, threads / 32);
  return launch_pdl(grouped_topk_fast_kernel<VPL>, dim3(blocks), dim3(threads), 0, s, gating, T, G, kg, k, scoring,
                    renorm, rsf, w, ids, z);
}

template <int VPL>
moe_status_t launch_topk(const float* gating, int T, int E, int G, int kg, int k, int scoring, int renorm, float rsf,
                         float* w, int32_t* ids, const RouteZero& z, cudaStream_t s) {
  const int threads = 256;
  const int blocks = cdiv(T, threads / 32);
  return launch_pdl(grouped_topk_kernel<VPL>, dim3(blocks), dim3(threads), 0, s, gating, T, E, G, kg, k, scoring,
                    renorm, rsf, w, ids, z);
}

// Thread-per-token kernel instances: (E, G, topk_group) with topk = 8.
template <int E, int G, int KG>
moe_status_t launch_tpt(const float* gating, int T, int scoring, int renorm, float rsf, float* w, int32_t* ids,
                        cudaStream_t s, int* err = nullptr, int32_t* tile_hist = nullptr) {
  CUtensorMap map;
  if (!make_tmap_f32_32x32(&map, gating, static_cast<uint64_t>(T), E)) return MOE_ERR_CUDA;
  auto kernel = tpt::grouped_topk_tpt_kernel<E, G, KG>;
  constexpr int smem = tpt::Shape<E>::kSmem;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kernel), smem)) return MOE_ERR_CUDA;
  const int ntiles = cdiv(T, tpt::kTile);
  const int sms = num_sms() > 0 ? num_sms() : 148;
  const int grid = ntiles < sms ? ntiles : sms;
  return launch_pdl(kernel, dim3(grid), dim3(tpt::kThreads), smem, s, map, T, ntiles, scoring, renorm, rsf, w, ids,
                    err, tile_hist);
}

bool tpt_applies(int T, int E, int G, int kg, int k, const void* w, const void* ids) {
  if (k != 8 || T < kTptMinTokens || !aligned16(w) || !aligned16(ids)) return false;
  return (E == 256 && G == 8 && kg == 4) || (E == 256 && G == 1) || (E == 128 && G == 1);
}

}  // namespace

// Routing that also writes the expert counts of every run of *tokens_per_row consecutive
// tokens (rows of E int32 at tile_hist: align's first pass over those pairs): the
// streaming kernel's 32-token tiles, or the segmented kernel's CTAs (rows_out rows).
// *rows_out = 0 (nothing launched) for the shapes of the other kernels, and the caller
// routes and counts the usual way. zero_rows / zero_cols: as for launch_grouped_topk
// (segmented kernel only).
moe_status_t launch_grouped_topk_tile_hist(const float* gating, int T, int E, int G, int kg, int k, int scoring,
                                           int renorm, float rsf, float* w, int32_t* ids, int32_t* tile_hist,
                                           int* err, float* zero_rows, int zero_cols, int* rows_out,
                                           int* tokens_per_row, cudaStream_t s) {
  *rows_out = 0;
  if (T == 0) return MOE_OK;
  if (!zero_rows && tpt_applies(T, E, G, kg, k, w, ids)) {
    *rows_out = cdiv(T, tpt::kTile);
    *tokens_per_row = tpt::kTile;
    if (E == 256 && G == 8) return launch_tpt<256, 8, 4>(gating, T, scoring, renorm, rsf, w, ids, s, err, tile_hist);
    if (E == 256) return launch_tpt<256, 1, 1>(gating, T, scoring, renorm, rsf, w, ids, s, err, tile_hist);
    return launch_tpt<128, 1, 1>(gating, T, scoring, renorm, rsf, w, ids, s, err, tile_hist);
  }
  const int L = (G & (G - 1)) == 0 ? seg_lanes(E, G, k) : 0;
  if (L == 0) return MOE_OK;
  const RouteZero z{reinterpret_cast<float4*>(zero_rows), zero_cols / 4, nullptr, 0, tile_hist, err};
  *tokens_per_row = kSegThreads / L;
  *rows_out = cdiv(T, kSegThreads / L);
  const int P = E / L;
  if (L == 8) {
    if (P == 4) return launch_seg<4, 8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
    if (P == 8) return launch_seg<8, 8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
    if (P == 16) return launch_seg<16, 8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
    if (P == 32) return launch_seg<32, 8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  } else if (L == 16) {
    if (P == 16) return launch_seg<16, 16>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
    if (P == 32) return launch_seg<32, 16>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  } else if (L == 32) {
    if (P == 16) return launch_seg<16, 32>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
    if (P == 32) return launch_seg<32, 32>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  }
  *rows_out = 0;
  return MOE_OK;
}

// The rows of counts launch_grouped_topk_tile_hist writes for this problem (0: none), and
// the tokens of each row.
int route_hist_rows(int T, int E, int G, int kg, int k, const void* w, const void* ids, bool zero_rows,
                    int* tokens_per_row) {
  if (T == 0) return 0;
  if (!zero_rows && tpt_applies(T, E, G, kg, k, w, ids)) {
    *tokens_per_row = tpt::kTile;
    return cdiv(T, tpt::kTile);
  }
  const int L = (G & (G - 1)) == 0 ? seg_lanes(E, G, k) : 0;
  if (L == 0) return 0;
  const int P = E / L;
  const bool inst = (L == 8 && (P == 4 || P == 8 || P == 16 || P == 32)) || (L == 16 && (P == 16 || P == 32)) ||
                    (L == 32 && (P == 16 || P == 32));
  if (!inst) return 0;
  *tokens_per_row = kSegThreads / L;
  return cdiv(T, kSegThreads / L);
}

moe_status_t validate_routing(int T, int E, int G, int kg, int k, int scoring) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || G < 1 || G > 32 || E % G != 0) return MOE_ERR_INVALID_ARG;
  if (kg < 1 || kg > G) return MOE_ERR_INVALID_ARG;
  if (k < 1 || k > MOE_MAX_TOPK || k > kg * (E / G)) return MOE_ERR_INVALID_ARG;
  if (scoring != MOE_SCORE_SOFTMAX && scoring != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t launch_grouped_topk(const float* gating, int T, int E, int G, int kg, int k, int scoring, int renorm,
                                 float rsf, float* w, int32_t* ids, cudaStream_t s, float* zero_rows, int zero_cols,
                                 int* zero_cnt, int cnt_per_row) {
  if (T == 0) return MOE_OK;
  const RouteZero z{reinterpret_cast<float4*>(zero_rows), zero_cols / 4, zero_cnt, cnt_per_row, nullptr, nullptr};
  // the thread-per-token kernel: enough tokens to stream, no rows to clear, its shapes
  if (!zero_rows && !zero_cnt && tpt_applies(T, E, G, kg, k, w, ids)) {
    if (E == 256 && G == 8) return launch_tpt<256, 8, 4>(gating, T, scoring, renorm, rsf, w, ids, s);
    if (E == 256) return launch_tpt<256, 1, 1>(gating, T, scoring, renorm, rsf, w, ids, s);
    return launch_tpt<128, 1, 1>(gating, T, scoring, renorm, rsf, w, ids, s);
  }
  const int L = (G & (G - 1)) == 0 ? seg_lanes(E, G, k) : 0;
  if (L == 8) {
    switch (E / L) {
      case 4: return launch_seg<4, 8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 8: return launch_seg<8, 8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 16: return launch_seg<16, 8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 32: return launch_seg<32, 8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      default: break;
    }
  } else if (L == 16) {
    switch (E / L) {
      case 16: return launch_seg<16, 16>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 32: return launch_seg<32, 16>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      default: break;
    }
  } else if (L == 32) {
    switch (E / L) {
      case 16: return launch_seg<16, 32>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 32: return launch_seg<32, 32>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      default: break;
    }
  }
  const bool pow2_groups = (G & (G - 1)) == 0;
  if (pow2_groups) {
    switch (E) {
      case 32: return launch_fast<1>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 64: return launch_fast<2>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 128: return launch_fast<4>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 256: return launch_fast<8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 512: return launch_fast<16>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      case 1024: return launch_fast<32>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
      default: break;
    }
  }
  const int per_lane = cdiv(E, 32);
  if (per_lane <= 1) return launch_topk<1>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  if (per_lane <= 2) return launch_topk<2>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  if (per_lane <= 4) return launch_topk<4>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  if (per_lane <= 8) return launch_topk<8>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  if (per_lane <= 16) return launch_topk<16>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  return launch_topk<32>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
}

}  // namespace moe

extern "C" moe_status_t moe_grouped_topk(const float* gating, int T, int E, int num_expert_group, int topk_group,
                                         int topk, int scoring, int renormalize, float routed_scaling_factor,
                                         float* topk_weights, int32_t* topk_ids, void* stream) {
  const moe_status_t st = moe::validate_routing(T, E, num_expert_group, topk_group, topk, scoring);
  if (st != MOE_OK) return st;
  if (T > 0 && (!gating || !topk_weights || !topk_ids)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && !moe::aligned16(gating)) return MOE_ERR_UNSUPPORTED;
  return moe::launch_grouped_topk(gating, T, E, num_expert_group, topk_group, topk, scoring, renormalize,
                                  routed_scaling_factor, topk_weights, topk_ids, moe::as_stream(stream), nullptr, 0,
                                  nullptr, 0);
}
