// moe_fused_forward_noalloc: the fused MoE layer forward for callers that cannot
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a plug-in or backend that
// runs inside a host framework which owns every byte of device memory and hands
// out no workspace, or a latency-critical caller that cannot afford an
// allocation (cudaMalloc may synchronise the device). For them this entry point
// takes the scratch memory moe_fused_forward needs from a fixed array compiled
// into the library instead of from a caller-provided workspace.
//
// The array is a file-scope __device__ object of MOE_NOALLOC_SCRATCH_BYTES bytes:
// every GPU on which the library's device code is loaded holds it until the
// process exits. Its host-side name is only a stand-in, so the device address is
// looked up with cudaGetSymbolAddress (on the first call made while a device is
// current) and cached together with the CUDA context it belongs to; a call made
// under another context of that device (after cudaDeviceReset, say) looks it up
// again instead of using the old address.
//
// All calls share the one array and it keeps the previous call's contents.
// Nothing in it has to start at zero: every buffer the forward reads is written
// earlier in the same call (the fp32 accumulator is cleared by the forward's own
// kernel). The device error word at its start collects MOE_DEVERR_* bits across
// calls until moe_fused_forward_noalloc_check_error reads and clears it. Calls
// whose GPU work overlaps (on different streams or host threads) race on the
// array and must be serialised by the caller.
#include "common.cuh"

#include <cuda.h>

#include <mutex>

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct ScratchAddr {
  CUcontext ctx = nullptr;
  void* addr = nullptr;
};
ScratchAddr g_noalloc_addr[kMaxDevices];

// The current context, from the driver entry point the runtime hands out (no link
// against the driver library); null if it cannot be had.
CUcontext current_context() {
  using GetCurrent = CUresult (*)(CUcontext*);
  static GetCurrent fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<GetCurrent>(nullptr);
    return reinterpret_cast<GetCurrent>(p);
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_noalloc_scratch on the current device, looked up once per
// (device, context).
moe_status_t noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  ScratchAddr& c = g_noalloc_addr[dev];
  if (!c.addr || !ctx || c.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    c.addr = p;
    c.ctx = ctx;
  }
  *out = c.addr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_fused_forward_noalloc(const void* x, const float* gating, const void* w_gate_up,
                                                  const void* w_down, int T, int H, int I, int E,
                                                  int num_expert_group, int topk_group, int topk, int scoring,
                                                  int renormalize, float routed_scaling_factor, void* y,
                                                  float* topk_weights, int32_t* topk_ids, void* stream) {
  // the scratch this problem needs: the layout of the kernels that its size selects
  const size_t need = moe_fused_forward_workspace_size(T, H, I, E, topk);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const moe_status_t st = noalloc_scratch(&scratch);
  if (st != MOE_OK) return st;
  return moe_fused_forward(x, gating, w_gate_up, w_down, T, H, I, E, num_expert_group, topk_group, topk, scoring,
                           renormalize, routed_scaling_factor, y, topk_weights, topk_ids, scratch,
                           MOE_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" moe_status_t moe_fused_forward_noalloc_check_error(int* code, void* stream) {
  if (!code) return MOE_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const moe_status_t st = noalloc_scratch(&scratch);
  if (st != MOE_OK) return st;
  return moe_check_device_error(scratch, code, stream);
}
