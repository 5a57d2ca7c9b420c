// noalloc.cu — ds_moe_verify_forward_noalloc: the MoE verify step run on a scratch array
// that belongs to the library image instead of a caller-supplied workspace.
//
// Who needs it: callers that cannot allocate device memory when they make the call — a
// plain C host loop that embeds one layer and owns no device allocator, or a server whose
// device memory is fully committed to a pre-reserved pool (weights, KV cache), where a
// cudaMalloc would fail, or would synchronise the device in the middle of a decode step.
// This call allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// The scratch is one file-scope __device__ array of DS_NOALLOC_SCRATCH_BYTES per device.
// Its device address is resolved once per device, on the first call made with that device
// current (cudaGetSymbolAddress; under lazy module loading the runtime loads this library's
// kernels at that point), so that first call should come before any stream capture.
// Every call on a device shares the one array: calls whose work overlaps on the GPU (two
// streams, or two host threads) race on it and give wrong results. The launch sequence
// clears, on the call's stream, every word of the scratch that must start at zero, so what
// an earlier call left there does not matter. The kernels report a bounded wait that gave
// up, or a failed device check, in a status word at the start of the array;
// ds_noalloc_status() reads it. The resolved address is kept for the life of the process:
// a cudaDeviceReset() destroys the context that owns the array, after which this call must
// not be used again in the process.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[DS_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_scratch_setup;

// Device address of the scratch array on the current device, resolved on first use.
ds_status scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DS_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_scratch_setup);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();  // leave no sticky error for the caller's next runtime call
        return DS_ERR_CUDA;
      }
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return DS_OK;
}

}  // namespace

extern "C" ds_status ds_moe_verify_forward_noalloc(const ds_moe_layer* layer,
                                                   const uint16_t* x, int32_t R, uint16_t* y,
                                                   int32_t* topk_idx, float* topk_w,
                                                   ds_stream_t stream) {
  // Host-only size check first: a layer that needs more scratch than the array holds is
  // refused before any CUDA call.
  const size_t need = ds_moe_workspace_size(layer, R);
  if (need == 0)   // sizes the call refuses: its own host check gives the status, no CUDA call
    return ds_moe_verify_forward(layer, x, R, y, topk_idx, topk_w, nullptr, 0, stream);
  if (need > (size_t)DS_NOALLOC_SCRATCH_BYTES) return DS_ERR_WORKSPACE;
  void* scratch = nullptr;
  const ds_status st = scratch_of_current_device(&scratch);
  if (st != DS_OK) return st;
  return ds_moe_verify_forward(layer, x, R, y, topk_idx, topk_w, scratch,
                               (size_t)DS_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" ds_status ds_noalloc_status(ds_stream_t stream) {
  void* scratch = nullptr;
  const ds_status st = scratch_of_current_device(&scratch);
  if (st != DS_OK) return st;
  return ds_workspace_status(scratch, stream);
}
