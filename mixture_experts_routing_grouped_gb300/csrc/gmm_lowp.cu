// gmm_lowp: low-precision grouped GEMM (entry points; kernels follow).
#include "common.cuh"

extern "C" size_t gmm_lowp_workspace_size(int M, int K, int N, int E) {
  (void)M; (void)K; (void)N; (void)E;
  return moe::kWsHeader;
}

extern "C" moe_status_t gmm_lowp(const void* input, const void* weights, const float* scales_x,
                                 const float* scales_w, const int32_t* expert_offsets, const int32_t* expert_sizes,
                                 void* out, int M, int K, int N, int E, int in_dt, int out_dt, void* ws,
                                 size_t ws_bytes, void* stream) {
  (void)input; (void)weights; (void)scales_x; (void)scales_w; (void)expert_offsets; (void)expert_sizes;
  (void)out; (void)M; (void)K; (void)N; (void)E; (void)in_dt; (void)out_dt; (void)ws; (void)ws_bytes;
  (void)stream;
  return MOE_ERR_UNSUPPORTED;
}
