// Symmetric per-row quantisation (per token for activations, per output channel
// for a weight matrix viewed as [E*N, K]).
//
// Follows the low-precision GMM article (pwwt.cn), section 3.2: scale =
// absmax(row) / 127 and q = clamp(round(x / scale), -127, 127) for INT8; the
// FP8-e4m3 variant uses absmax / 448 and a round-to-nearest-even, saturating
// conversion. Scale and quotient are IEEE fp32 operations (no fast-math), so the
// codes are exactly those of the same arithmetic done on the host; the quotient is
// formed as x * RN(1/scale) wherever an error bound shows that gives the same code,
// else by the correctly rounded division. An all-zero row gets scale 1 and codes 0.
//
// Rows of up to 2048 bf16 (1024 fp32) values are loaded once into the registers
// of 8, 16 or 32 lanes (several rows per warp), and the absmax and the codes are
// computed from there; longer rows take one warp each and are read twice
// (absmax, then quantise), the second time mostly from L1/L2.
#include "common.cuh"

#include <cuda_fp8.h>

namespace moe {
namespace {

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Code of r, the fp32 quotient x / s, for one value.
template <bool E4M3>
__device__ __forceinline__ uint32_t code_of(float r) {
  if (E4M3) return static_cast<uint32_t>(__nv_cvt_float_to_fp8(r, __NV_SATFINITE, __NV_E4M3));
  const float rq = fminf(fmaxf(rintf(r), -127.f), 127.f);
  return static_cast<uint32_t>(static_cast<int>(rq)) & 0xffu;
}

// Whether y = x * RN(1/s) may round to another code than RN(x / s) does. With
// u = 2^-24, RN(1/s) = (1/s)(1 + e1) and y = (x/s)(1 + e1)(1 + e2), |e1|, |e2| <= u, so
// |y - x/s| < 2 ulp(x/s) and y, RN(x/s) are at most 2 ulps apart (one binade: the
// boundaries below sit mid-binade). The two codes can then differ only where a
// rounding boundary of the target lies within 2 ulps of y; the test takes 3.
//  e4m3, |y| >= 2^-6: the boundaries are the midpoints 2^e (1 + (2m+1)/16), whose fp32
//    encodings have bit 19 set and bits 18..0 clear; 0 < |y| < 2^-6 (e4m3 subnormals,
//    whose boundaries are spread over several binades) always takes the exact path.
//  INT8: the boundaries are the half-integers; |y - rint(y)| is exact, and 2^-14
//    exceeds 3 ulps for every |y| < 128.
template <bool E4M3>
__device__ __forceinline__ bool needs_exact(float y) {
  if (E4M3) {
    const uint32_t a = __float_as_uint(y) & 0x7fffffffu;
    return (a - 1u < 0x3c800000u - 1u) || ((a & 0xfffffu) - 0x7fffdu < 7u);
  }
  return fabsf(fabsf(y - rintf(y)) - 0.5f) <= 0x1p-14f;
}

// Per-row constants of the quotient: s, RN(1/s), and whether the product path is
// valid for the row (s and 1/s normal, so that neither rounding step underflows
// outside the e4m3 subnormal range, which is checked per value).
struct RowScale {
  float s, rs;
  bool exact;
};

__device__ __forceinline__ RowScale row_scale(float sc) {
  RowScale r;
  r.s = sc;
  r.rs = __frcp_rn(sc);
  r.exact = !(sc >= 0x1p-125f && sc <= 0x1p125f);
  return r;
}

// Codes of eight values x / s, packed little-endian: x * RN(1/s) where that is
// provably the same code, else the correctly rounded quotient for the whole chunk.
template <bool E4M3>
__device__ __forceinline__ uint2 quant_chunk(const float (&v)[8], const RowScale& rs) {
  float y[8];
  bool exact = rs.exact;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    y[j] = v[j] * rs.rs;
    exact |= needs_exact<E4M3>(y[j]);
  }
  if (exact) {
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = __fdiv_rn(v[j], rs.s);
  }
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    lo |= code_of<E4M3>(y[j]) << (8 * j);
    hi |= code_of<E4M3>(y[j + 4]) << (8 * j);
  }
  return make_uint2(lo, hi);
}

template <typename T, bool E4M3>
__global__ void __launch_bounds__(256) quant_rows_kernel(const T* __restrict__ x, int M, int K,
                                                         uint8_t* __restrict__ q, float* __restrict__ scales,
                                                         const int* __restrict__ rows_dev) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= M || (rows_dev && row >= __ldg(rows_dev))) return;
  const T* xr = x + static_cast<size_t>(row) * K;
  float amax = 0.f;
  for (int c = lane * 8; c < K; c += 256) {
    float v[8];
    load8<T>(xr + c, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float qmax = E4M3 ? 448.0f : 127.0f;
  const float s = (amax == 0.f) ? 1.0f : __fdiv_rn(amax, qmax);
  if (lane == 0) scales[row] = s;
  const RowScale rs = row_scale(s);
  uint8_t* qr = q + static_cast<size_t>(row) * K;
  for (int c = lane * 8; c < K; c += 256) {
    float v[8];
    load8<T>(xr + c, v);
    *reinterpret_cast<uint2*>(qr + c) = quant_chunk<E4M3>(v, rs);
  }
}

// Raw 16-byte chunks of 8 values: bf16 rows keep one uint4 per chunk, fp32 rows two.
template <typename T> struct Chunk;
template <> struct Chunk<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void values(float (&v)[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};
template <> struct Chunk<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void values(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// Register-resident variant: L lanes per row (32 / L rows per warp), lane s of a
// row holding its chunks s + L i (i < C) in registers, K <= 8 L C. All of a
// lane's loads are in flight together and the row is read once; a row's chain
// (loads, absmax, L-lane reduction, scale, codes) is short enough, and there are
// enough rows per warp, that the kernel streams instead of waiting on one
// row's latency per warp.
template <typename T, bool E4M3, int L, int C>
__global__ void __launch_bounds__(256) quant_rows_reg_kernel(const T* __restrict__ x, int M, int K,
                                                             uint8_t* __restrict__ q, float* __restrict__ scales,
                                                             const int* __restrict__ rows_dev) {
  const int gl = blockIdx.x * blockDim.x + threadIdx.x;
  const int row = gl / L;
  const int sub = gl & (L - 1);
  const int m = rows_dev ? min(M, __ldg(rows_dev)) : M;
  const bool live = row < m;
  const T* xr = x + static_cast<size_t>(live ? row : 0) * K;
  Chunk<T> raw[C];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int c = (sub + L * i) * 8;
    if (live && c < K) raw[i].load(xr + c);
  }
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int c = (sub + L * i) * 8;
    if (live && c < K) {
      float v[8];
      raw[i].values(v);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
    }
  }
#pragma unroll
  for (int o = 1; o < L; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (!live) return;
  const float qmax = E4M3 ? 448.0f : 127.0f;
  const float sc = (amax == 0.f) ? 1.0f : __fdiv_rn(amax, qmax);
  if (sub == 0) scales[row] = sc;
  const RowScale rs = row_scale(sc);
  uint8_t* qr = q + static_cast<size_t>(row) * K;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int c = (sub + L * i) * 8;
    if (c < K) {
      float v[8];
      raw[i].values(v);
      *reinterpret_cast<uint2*>(qr + c) = quant_chunk<E4M3>(v, rs);
    }
  }
}

template <typename T, bool E4M3, int L, int C>
void launch_reg(const T* x, int M, int K, uint8_t* q, float* s, cudaStream_t st, const int* rows_dev) {
  const int rows_per_block = 256 / L;
  quant_rows_reg_kernel<T, E4M3, L, C><<<cdiv(M, rows_per_block), 256, 0, st>>>(x, M, K, q, s, rows_dev);
}

// Lanes per row: the fewest (>= 8) that keep a lane's chunks within C (8 for bf16
// rows, 4 for fp32 rows: 32 registers of raw data, so that enough warps stay
// resident to hide each row's dependent chain); rows longer than 32 lanes' worth
// take the two-pass kernel.
template <typename T, bool E4M3>
void launch_quant_t(const T* x, int M, int K, uint8_t* q, float* s, cudaStream_t st, const int* rows_dev) {
  constexpr int C = sizeof(T) == 2 ? 8 : 4;
  if (K <= 8 * 8 * C) launch_reg<T, E4M3, 8, C>(x, M, K, q, s, st, rows_dev);
  else if (K <= 8 * 16 * C) launch_reg<T, E4M3, 16, C>(x, M, K, q, s, st, rows_dev);
  else if (K <= 8 * 32 * C) launch_reg<T, E4M3, 32, C>(x, M, K, q, s, st, rows_dev);
  else quant_rows_kernel<T, E4M3><<<cdiv(M, 8), 256, 0, st>>>(x, M, K, q, s, rows_dev);
}

template <typename T>
void launch_quant(const void* x, int M, int K, bool e4m3, void* q, float* s, cudaStream_t st,
                  const int* rows_dev = nullptr) {
  if (e4m3)
    launch_quant_t<T, true>(static_cast<const T*>(x), M, K, static_cast<uint8_t*>(q), s, st, rows_dev);
  else
    launch_quant_t<T, false>(static_cast<const T*>(x), M, K, static_cast<uint8_t*>(q), s, st, rows_dev);
}

}  // namespace

// Per-row e4m3 quantisation of a bf16 matrix for the fused FP8 forward: rows at
// or past *rows_dev (read on the device) are left untouched.
moe_status_t launch_quant_rows_e4m3_bf16(const __nv_bfloat16* x, int M, int K, uint8_t* q, float* s,
                                         const int* rows_dev, cudaStream_t st) {
  if (M == 0) return MOE_OK;
  launch_quant<__nv_bfloat16>(x, M, K, true, q, s, st, rows_dev);
  return launch_status();
}

}  // namespace moe

extern "C" moe_status_t moe_quant_per_token(const void* x, int x_dt, int M, int K, int q_dt, void* q,
                                            float* scales, void* stream) {
  if (M < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (x_dt != MOE_DT_BF16 && x_dt != MOE_DT_F32) return MOE_ERR_INVALID_ARG;
  if (q_dt != MOE_DT_I8 && q_dt != MOE_DT_E4M3) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!x || !q || !scales)) return MOE_ERR_INVALID_ARG;
  if (K % 8 != 0 || (M > 0 && (!moe::aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7u) != 0)))
    return MOE_ERR_UNSUPPORTED;
  if (M == 0) return MOE_OK;
  cudaStream_t s = moe::as_stream(stream);
  if (x_dt == MOE_DT_BF16)
    moe::launch_quant<__nv_bfloat16>(x, M, K, q_dt == MOE_DT_E4M3, q, scales, s);
  else
    moe::launch_quant<float>(x, M, K, q_dt == MOE_DT_E4M3, q, scales, s);
  return moe::launch_status();
}
