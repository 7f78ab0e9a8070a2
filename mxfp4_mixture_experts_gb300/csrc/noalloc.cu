// mxfp4_moe_forward_noalloc: the forward call for callers that cannot
// allocate device memory. Its workspace is a fixed array compiled into this
// library (see include/mxfp4_moe.h for the contract); everything else is the
// ordinary mxfp4_moe_forward, called unchanged.
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "../../include/mxfp4_moe.h"
#include "kernels.h"

namespace {

// Workspace of the no-allocation entry point. Every GPU that loads the
// library holds it until the process exits. Static storage starts zeroed.
static __device__ __align__(256) unsigned char g_noalloc_ws[MXFP4_MOE_NOALLOC_BYTES];

constexpr int kMaxDevices = 64;
void* g_ws[kMaxDevices] = {};
std::mutex g_mu;

// Host code cannot use g_noalloc_ws directly (that name is a host-side stand-in,
// not a device address): ask the runtime for the device address, once per
// device, with that device current.
int noalloc_workspace(void** ws, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXFP4_MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_ws[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr)
      return MXFP4_MOE_ERR_CUDA;
    // the first bytes of any workspace hold counters that must be zero when a
    // call starts; every call leaves them zero again, also one whose bounded
    // wait gave up, so they are cleared once, here
    const size_t zero_kept = mxmoe::workspace_zero_kept_bytes();
    if (zero_kept > sizeof(g_noalloc_ws)) return MXFP4_MOE_ERR_WORKSPACE;
    if (cudaMemsetAsync(p, 0, zero_kept, stream) != cudaSuccess) return MXFP4_MOE_ERR_CUDA;
    g_ws[dev] = p;
  }
  *ws = g_ws[dev];
  return MXFP4_MOE_OK;
}

}  // namespace

extern "C" int mxfp4_moe_forward_noalloc(const void* hidden, const int32_t* topk_ids,
                                         const float* topk_weights, const uint8_t* w13,
                                         const uint8_t* s13, const uint8_t* w2,
                                         const uint8_t* s2, int T, int K, int I, int E,
                                         int topk, void* out, int32_t* status, int path,
                                         void* stream) {
  const size_t need = mxfp4_moe_workspace_size(T, K, I, E, topk);
  if (need == 0) return MXFP4_MOE_ERR_SHAPE;
  if (need > (size_t)MXFP4_MOE_NOALLOC_BYTES) return MXFP4_MOE_ERR_WORKSPACE;
  if (T == 0) return MXFP4_MOE_OK;
  void* ws = nullptr;
  if (int rc = noalloc_workspace(&ws, static_cast<cudaStream_t>(stream))) return rc;
  return mxfp4_moe_forward(hidden, topk_ids, topk_weights, w13, s13, w2, s2, T, K, I, E, topk,
                           out, status, ws, (size_t)MXFP4_MOE_NOALLOC_BYTES, path, stream);
}
