// common.cuh — device helpers shared by the kernels of libdsmoe.so (sm_103a).
#pragma once
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dsmoe.h"

namespace dsmoe {

// Bits of the device status word kept in a workspace header (read by ds_workspace_status).
enum : uint32_t {
  kStatusTimeout = 1u,      // a bounded wait gave up
  kStatusCheck = 2u,        // a consistency / bounds check failed (access skipped)
};

// Workspace header: first 256 bytes of every workspace, zeroed at the start of each call.
struct WsHeader {
  uint32_t status;
  uint32_t router_arrivals;   // K1 last-CTA hand-off counter
  uint32_t reserved[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Programmatic dependent launch: a grid launched with launch_pdl may start while the grid
// before it in the stream finishes; pdl_wait() returns once that grid has completed and its
// memory operations are visible. pdl_trigger() lets the next grid start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Exp, typename... Act>
cudaError_t launch_pdl(void (*kernel)(Exp...), dim3 grid, int block, size_t smem, cudaStream_t s,
                       Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

__device__ __forceinline__ void flag_status(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}
// Low / high bf16 of a packed pair widened to fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  // Weight bytes are read exactly once per call: keep them out of L1.
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

}  // namespace dsmoe
