// Shared host/device helpers of the MoE library (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstddef>

#include "moe_gb300.h"

namespace moe {

constexpr int kWarp = 32;

// Workspace header: the first 256 bytes of every workspace.
//   [0]   int32 device error word (MOE_DEVERR_* bits)
//   [4..] int32 scratch counters used by the kernels of one call
constexpr size_t kWsHeader = 256;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Records a device-side data error without trapping.
__device__ inline void report_error(int* err, int bits) {
  if (err) atomicOr(err, bits);
}

// Number of SMs of the current device (cached per device).
int num_sms();

moe_status_t launch_status();

// Raises a kernel's dynamic shared memory limit to at least `bytes` (the largest
// limit set so far is remembered per (kernel, device)).
bool ensure_smem_attr(const void* func, int bytes);

// Programmatic dependent launch. Every kernel of the layer is launched as a
// programmatic dependent of the kernel before it in the stream (launch_pdl): it may
// start while that kernel finishes, so its launch, and the on-chip set-up done before
// pdl_wait, overlap the other's tail. pdl_wait returns once the kernel before it has
// completed with its memory visible; no kernel touches global memory before it. Each
// kernel calls pdl_trigger first, so that its own dependent may be scheduled as soon
// as all of its CTAs have started (the dependent's CTAs then wait in pdl_wait).
// Outside such a launch both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline moe_status_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_status();
}

}  // namespace moe
