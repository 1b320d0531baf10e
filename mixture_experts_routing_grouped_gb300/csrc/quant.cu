// Symmetric per-row quantisation (per token for activations, per output channel
// for a weight matrix viewed as [E*N, K]).
//
// Follows the low-precision GMM article (pwwt.cn), section 3.2: scale =
// absmax(row) / 127 and q = clamp(round(x / scale), -127, 127) for INT8; the
// FP8-e4m3 variant uses absmax / 448 and a round-to-nearest-even, saturating
// conversion. Scale and quotient are IEEE fp32 operations (no fast-math), so the
// codes are exactly those of the same arithmetic done on the host. An all-zero
// row gets scale 1 and codes 0.
//
// One warp per row; the row is read twice (absmax, then quantise), the second
// time mostly from L1/L2.
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
  uint8_t* qr = q + static_cast<size_t>(row) * K;
  for (int c = lane * 8; c < K; c += 256) {
    float v[8];
    load8<T>(xr + c, v);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float r = __fdiv_rn(v[i], s);
      uint32_t code;
      if (E4M3) {
        code = static_cast<uint32_t>(__nv_cvt_float_to_fp8(r, __NV_SATFINITE, __NV_E4M3));
      } else {
        const float rq = fminf(fmaxf(rintf(r), -127.f), 127.f);
        code = static_cast<uint32_t>(static_cast<int>(rq)) & 0xffu;
      }
      if (i < 4) lo |= code << (8 * i); else hi |= code << (8 * (i - 4));
    }
    *reinterpret_cast<uint2*>(qr + c) = make_uint2(lo, hi);
  }
}

template <typename T>
void launch_quant(const void* x, int M, int K, bool e4m3, void* q, float* s, cudaStream_t st,
                  const int* rows_dev = nullptr) {
  const int threads = 256;
  const int blocks = cdiv(M, threads / 32);
  if (e4m3)
    quant_rows_kernel<T, true><<<blocks, threads, 0, st>>>(static_cast<const T*>(x), M, K,
                                                            static_cast<uint8_t*>(q), s, rows_dev);
  else
    quant_rows_kernel<T, false><<<blocks, threads, 0, st>>>(static_cast<const T*>(x), M, K,
                                                             static_cast<uint8_t*>(q), s, rows_dev);
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
