// Allocation-free variant of the decode block: the per-call workspace lives in
// a fixed device array compiled into this library instead of memory the
// caller allocates.
//
// Who needs it: callers that cannot call cudaMalloc at the point where they
// run a decode step -- for example code running under a memory-pool or
// allocation-hook policy that forbids new device allocations after start-up,
// plugin hosts that hand the library only input/output buffers, or latency-
// critical loops where an allocation (and its implicit synchronisation) is not
// acceptable.  They still pass the weights, cache, inputs and outputs; only
// the scratch space comes from here.
//
// Properties a caller must know:
//  * the array is kStaticWorkspaceBytes (48 MiB) of device memory that every GPU
//    loading this library keeps until the process exits (the largest layer
//    shape here, 70B at batch 32, needs about 33 MiB);
//  * problems whose workspace would exceed it are rejected with
//    FT_ERR_WORKSPACE before anything is enqueued;
//  * the array is shared by every call on a device and keeps the previous
//    call's contents; everything the block needs zeroed is cleared by its own
//    first kernel, so no clearing is required between calls, but calls that
//    overlap on the GPU (different streams, or different host threads without
//    ordering) race on the array and produce wrong results;
//  * the device address of the array is looked up with cudaGetSymbolAddress
//    the first time the entry point runs on each device (with that device
//    current); make that first call before any stream capture begins.  The
//    address is kept for the life of the process, so the entry point must not
//    be used on a device after cudaDeviceReset (or any other teardown of its
//    primary context) in the same process.
#include <mutex>

#include "ft_internal.cuh"

namespace {

constexpr size_t kStaticWorkspaceBytes = 48u << 20;

// Device-side scratch.  In host code this name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_ws_mu;
void* g_ws_ptr[64] = {nullptr};

int static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FT_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (!g_ws_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return FT_ERR_CUDA;
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return FT_OK;
}

}  // namespace

extern "C" {

int ft_decode_block_static_ws(const ft_block_cfg* c, const ft_layer_weights* w, void* cache, int max_batch,
                              int max_ctx, const void* x_in, void* x_out, int act_dtype, const int32_t* pos, int B,
                              int32_t* dev_status, ft_stream stream) {
  const int e = ft_host::check_cfg(c);
  if (e != FT_OK) return e;
  if (B > 32) return FT_ERR_UNSUPPORTED;
  if (B < 1 || max_ctx < 1) return FT_ERR_INVALID_ARG;
  const size_t need = ft_decode_workspace_bytes(c, B, max_ctx);
  if (need == 0) return FT_ERR_INVALID_ARG;
  if (need > kStaticWorkspaceBytes) return FT_ERR_WORKSPACE;
  void* ws = nullptr;
  const int s = static_workspace(&ws);
  if (s != FT_OK) return s;
  return ft_decode_block(c, w, cache, max_batch, max_ctx, x_in, x_out, act_dtype, pos, B, ws, kStaticWorkspaceBytes,
                         dev_status, stream);
}

}  // extern "C"
