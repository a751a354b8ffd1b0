// noalloc.cu -- dab_attn_bwd_noalloc: the attention backward for callers that
// cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc at the point where they
// need the backward: a plugin running inside a host framework that owns and
// budgets all device memory, or a latency-critical loop where an allocation
// (which may synchronise the device) is not acceptable.  For them the
// workspace of dab_attn_bwd (status word, dispatch counter, semaphores, D,
// LSE*log2(e) and the f32 dQ accumulator) lives in one file-scope device
// array of a fixed size instead of caller-provided memory.  Every GPU that
// loads the library holds this array until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "dab.h"

namespace {

constexpr size_t kScratchBytes = DAB_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch array.  In host code its name is only a host-side stand-in for
// the device symbol, never a device address: a kernel handed the name would
// fault or, where the GPU can reach host memory, silently use the wrong
// memory.  Host code passes the address that cudaGetSymbolAddress returns.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: look up the device address of
// the scratch array.  Returns nullptr if the lookup failed.  The address is
// kept for the life of the process; a cudaDeviceReset() unloads the module
// that holds the array, so this entry point must not be used on a device
// after it has been reset.
void* scratch_for_current_device(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" dab_status_t dab_noalloc_check_status(cudaStream_t stream) {
  int dev = -1;
  void* scratch = scratch_for_current_device(&dev);
  if (scratch == nullptr) return DAB_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DAB_ERR_CUDA;
  // The status and detail words head the array (offset 0 of the workspace
  // layout); copied into host stack memory, nothing is allocated.
  uint32_t hdr[2] = {0u, 0u};
  if (cudaMemcpyFromSymbol(hdr, g_scratch, sizeof(hdr), 0, cudaMemcpyDeviceToHost) != cudaSuccess)
    return DAB_ERR_CUDA;
  if (hdr[0] == 0u) return DAB_OK;
  if (hdr[0] == DAB_ERR_TIMEOUT || hdr[0] == DAB_ERR_DEVICE_BOUNDS) return (dab_status_t)hdr[0];
  return DAB_ERR_DEVICE_BOUNDS;
}

extern "C" dab_status_t dab_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                             const void* o, const float* lse, const void* dout,
                                             void* dq, void* dk, void* dv, int B, int H, int S,
                                             int d, float scale, dab_mask_t mask,
                                             dab_sched_t sched, cudaStream_t stream) {
  const size_t need = dab_bwd_workspace_size(B, H, S, d, mask, sched);
  if (need == 0) return DAB_ERR_INVALID_ARG;  // invalid shape or enum
  if (need > kScratchBytes) return DAB_ERR_WORKSPACE;  // beyond the built-in maximum
  int dev = -1;
  void* scratch = scratch_for_current_device(&dev);
  if (scratch == nullptr) return DAB_ERR_CUDA;
  // The ordinary path, on the built-in scratch.  Its first kernel resets
  // everything that must start at zero (status word, dispatch counter,
  // semaphores, and for ATOMIC the accumulator), so the previous call's
  // contents do no harm.
  return dab_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, S, d, scale, mask, sched, scratch,
                      kScratchBytes, stream);
}
