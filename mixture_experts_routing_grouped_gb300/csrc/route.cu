// Grouped top-k routing: one warp per token, everything in registers.
//
// Follows "GroupedTopK 算子优化入门" section 三 (score, per-group max, top
// groups, mask, top-k, renormalise, scale) with the fusion plan of its
// section 六 (one program per token, only the k weights and k ids are written)
// and the simplification of section 七: both score functions are strictly
// increasing, so groups and experts are selected on the logits themselves and
// only the k selected logits are exponentiated when the weights renormalise.
//
// Lane l holds the logits of experts [l*VPL, (l+1)*VPL). Warp-wide maxima and
// the lowest index among equal maxima come from redux.sync, so ties resolve to
// the lower expert (or group) index. The fast kernel (E = 32*VPL, power-of-two
// group count) reduces the float logits directly; the generic kernel (any E and
// G) reduces order-preserving unsigned keys of the logits.
#include "common.cuh"

#include <cuda_runtime.h>
#include <math_constants.h>

namespace moe {
namespace {

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

template <int VPL>
void launch_fast(const float* gating, int T, int G, int kg, int k, int scoring, int renorm, float rsf, float* w,
                 int32_t* ids, const RouteZero& z, cudaStream_t s) {
  const int threads = 256;
  const int blocks = cdiv(T, threads / 32);
  grouped_topk_fast_kernel<VPL><<<blocks, threads, 0, s>>>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z);
}

template <int VPL>
void launch_topk(const float* gating, int T, int E, int G, int kg, int k, int scoring, int renorm, float rsf,
                 float* w, int32_t* ids, const RouteZero& z, cudaStream_t s) {
  const int threads = 256;
  const int blocks = cdiv(T, threads / 32);
  grouped_topk_kernel<VPL><<<blocks, threads, 0, s>>>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z);
}

}  // namespace

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
  const RouteZero z{reinterpret_cast<float4*>(zero_rows), zero_cols / 4, zero_cnt, cnt_per_row};
  const bool pow2_groups = (G & (G - 1)) == 0;
  if (pow2_groups) {
    switch (E) {
      case 32: launch_fast<1>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s); return launch_status();
      case 64: launch_fast<2>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s); return launch_status();
      case 128: launch_fast<4>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s); return launch_status();
      case 256: launch_fast<8>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s); return launch_status();
      case 512: launch_fast<16>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s); return launch_status();
      case 1024: launch_fast<32>(gating, T, G, kg, k, scoring, renorm, rsf, w, ids, z, s); return launch_status();
      default: break;
    }
  }
  const int per_lane = cdiv(E, 32);
  if (per_lane <= 1) launch_topk<1>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  else if (per_lane <= 2) launch_topk<2>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  else if (per_lane <= 4) launch_topk<4>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  else if (per_lane <= 8) launch_topk<8>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  else if (per_lane <= 16) launch_topk<16>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  else launch_topk<32>(gating, T, E, G, kg, k, scoring, renorm, rsf, w, ids, z, s);
  return launch_status();
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
