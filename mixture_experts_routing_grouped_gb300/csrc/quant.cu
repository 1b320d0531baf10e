// Symmetric per-row quantisation (per token for activations, per output channel
// for a weight matrix viewed as [E*N, K]).
//
// Follows the low-precision GMM article (pwwt.cn), section 3.2: scale =
// absmax(row) / 127 and q = clamp(round(x / scale), -127, 127) for INT8; the
// FP8-e4m3 variant uses absmax / 448 and a round-to-nearest-even, saturating
// conversion. Scale and quotient are IEEE fp32 operations (no fast-math), so the
// codes are exactly those of the same arithmetic done on the host; the quotient is
// bracketed by two products x * RN(1/scale) (1 -+ 2^-21), whose codes, where they
// agree, are provably the code of the correctly rounded quotient; elsewhere it is
// the correctly rounded division. An all-zero row gets scale 1 and codes 0.
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

// Per-row constants of the quotient. With u = 2^-24 and r = RN(1/s), the bracket
// factors are r_lo = RN(r (1 - 8u)) and r_hi = RN(r (1 + 8u)); for z = x / s > 0,
//   RN(x r_lo) <= z (1 + u)^3 (1 - 8u) < z (1 - u) <= RN(z)
// and symmetrically RN(x r_hi) > RN(z) (mirrored for z < 0), each step a correctly
// rounded fp32 operation of relative error at most u. Both codes (e4m3 round to
// nearest even with saturation, and INT8 rint then clamp) are monotone in their
// argument, so where the codes of RN(x r_lo) and RN(x r_hi) agree they are the code of
// RN(z). Where they differ, a rounding boundary M lies between the two; if x = M s
// exactly (fma(-M, s, x) == 0, no underflow for the rows' range of s) then RN(z) = M,
// whose own conversion settles the tie; otherwise the value takes the correctly
// rounded division. Rows with s outside [2^-100, 2^100] take the division throughout.
// Below the fp32 normal range every bracket value and RN(z) has code +-0 with the
// sign of x.
struct RowScale {
  float s, lo, hi;
  bool exact;
};

__device__ __forceinline__ RowScale row_scale(float sc) {
  RowScale r;
  const float rc = __frcp_rn(sc);
  r.s = sc;
  r.lo = rc * (1.0f - 0x1p-21f);
  r.hi = rc * (1.0f + 0x1p-21f);
  r.exact = !(sc >= 0x1p-100f && sc <= 0x1p100f);
  return r;
}

// Codes of two values x / s (value 0 in the low byte) from the bracket alone, and a
// flag set where either value's bracket codes differ or the row takes the division.
template <bool E4M3>
__device__ __forceinline__ uint32_t quant_pair_fast(float x0, float x1, const RowScale& rs, bool& flag) {
  const float a0 = x0 * rs.lo, a1 = x1 * rs.lo;
  const float b0 = x0 * rs.hi, b1 = x1 * rs.hi;
  if (E4M3) {
    const uint32_t cl = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
    flag = rs.exact || cl != __nv_cvt_float2_to_fp8x2(make_float2(b0, b1), __NV_SATFINITE, __NV_E4M3);
    return cl;
  }
  const float l0 = rintf(a0), l1 = rintf(a1);
  flag = rs.exact || l0 != rintf(b0) || l1 != rintf(b1);
  return code_of<false>(l0) | (code_of<false>(l1) << 8);
}

// Codes of eight values, packed little-endian (value j in byte j); bit p of the
// returned flags marks pair p (values 2p, 2p+1) for resolve_pair.
template <bool E4M3>
__device__ __forceinline__ uint2 quant_chunk_fast(const float (&v)[8], const RowScale& rs, uint32_t& flags) {
  uint32_t c[4];
  flags = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    bool f;
    c[p] = quant_pair_fast<E4M3>(v[2 * p], v[2 * p + 1], rs, f);
    flags |= static_cast<uint32_t>(f) << p;
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Exact code of one value x / s. Where the bracket codes differ, M is the boundary
// between them: for e4m3 the bracket's low end rounded to 4 fractional mantissa bits
// (every e4m3 midpoint has at most that many), for INT8 the half-integer between the
// two. x = M s exactly (fma(-M, s, x) == 0) makes RN(x / s) = M, whose conversion
// settles the tie; anything else takes the correctly rounded division.
template <bool E4M3>
__device__ __forceinline__ uint32_t code_exact(float x, const RowScale& rs) {
  const float a = x * rs.lo, b = x * rs.hi;
  float m;
  if (E4M3) m = __uint_as_float((__float_as_uint(a) + 0x40000u) & 0xfff80000u);
  else m = (rintf(a) + rintf(b)) * 0.5f;
  if (!rs.exact) {
    const uint32_t ca = code_of<E4M3>(a);
    if (ca == code_of<E4M3>(b)) return ca;
    if (fmaf(-m, rs.s, x) == 0.0f) return code_of<E4M3>(m);
  }
  return code_of<E4M3>(__fdiv_rn(x, rs.s));
}

template <typename T>
__device__ __forceinline__ void load2(const T* p, float& v0, float& v1);
template <>
__device__ __forceinline__ void load2<float>(const float* p, float& v0, float& v1) {
  const float2 a = __ldg(reinterpret_cast<const float2*>(p));
  v0 = a.x;
  v1 = a.y;
}
template <>
__device__ __forceinline__ void load2<__nv_bfloat16>(const __nv_bfloat16* p, float& v0, float& v1) {
  const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
  v0 = __uint_as_float(w << 16);
  v1 = __uint_as_float(w & 0xffff0000u);
}

// Rewrites the two codes at column c (even) of a row whose fast codes were stored
// earlier by this thread, re-reading the two values (cached).
template <typename T, bool E4M3>
__device__ __forceinline__ void resolve_pair(const T* xr, uint8_t* qr, int c, const RowScale& rs) {
  float v0, v1;
  load2<T>(xr + c, v0, v1);
  const uint32_t code = code_exact<E4M3>(v0, rs) | (code_exact<E4M3>(v1, rs) << 8);
  *reinterpret_cast<uint16_t*>(qr + c) = static_cast<uint16_t>(code);
}

template <typename T, bool E4M3>
__global__ void __launch_bounds__(256) quant_rows_kernel(const T* __restrict__ x, int M, int K,
                                                         uint8_t* __restrict__ q, float* __restrict__ scales,
                                                         const int* __restrict__ rows_dev) {
  pdl_trigger();
  pdl_wait();
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
    uint32_t f;
    *reinterpret_cast<uint2*>(qr + c) = quant_chunk_fast<E4M3>(v, rs, f);
    while (f) {
      const int p = __ffs(f) - 1;
      f &= f - 1;
      resolve_pair<T, E4M3>(xr, qr, c + 2 * p, rs);
    }
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
  pdl_trigger();
  pdl_wait();
  static_assert(4 * C <= 32, "one flag bit per pair of a lane's chunks");
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
  uint32_t flagged = 0;  // bit 4 i + p: pair p of chunk i needs resolve_pair
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int c = (sub + L * i) * 8;
    if (c < K) {
      float v[8];
      raw[i].values(v);
      uint32_t f;
      *reinterpret_cast<uint2*>(qr + c) = quant_chunk_fast<E4M3>(v, rs, f);
      flagged |= f << (4 * i);
    }
  }
  // One copy of the exact path, outside the unrolled loop: rare pairs only.
  while (flagged) {
    const int b = __ffs(flagged) - 1;
    flagged &= flagged - 1;
    resolve_pair<T, E4M3>(xr, qr, (sub + L * (b >> 2)) * 8 + 2 * (b & 3), rs);
  }
}

template <typename T, bool E4M3, int L, int C>
void launch_reg(const T* x, int M, int K, uint8_t* q, float* s, cudaStream_t st, const int* rows_dev) {
  const int rows_per_block = 256 / L;
  (void)launch_pdl(quant_rows_reg_kernel<T, E4M3, L, C>, dim3(cdiv(M, rows_per_block)), dim3(256), 0, st, x, M, K, q,
                   s, rows_dev);
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
  else (void)launch_pdl(quant_rows_kernel<T, E4M3>, dim3(cdiv(M, 8)), dim3(256), 0, st, x, M, K, q, s, rows_dev);
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
