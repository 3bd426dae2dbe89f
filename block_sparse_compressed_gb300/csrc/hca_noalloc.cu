// hca_noalloc.cu -- hca_attn_fwd_noalloc: the forward pass with built-in
// scratch, for callers that must not allocate device memory.
//
// Who needs it.  Some callers have no way to hand over device scratch at the
// moment they run attention: plugin "enqueue" hooks of inference runtimes
// that forbid device allocation inside the call, real-time loops where
// cudaMalloc's implicit synchronisation would stall the pipeline, and plain C
// hosts that own no allocator at all.  This entry point lets them run the
// forward with only their inputs and outputs.
//
// How.  The scratch the forward needs (a status word and one int32 per
// position for the document starts) lives in a file-scope __device__ array
// of fixed size.  Every GPU that loads libhca holds that array until the
// process exits.  Host code cannot use the array's name as a device address,
// so the first call on each device (with that device current) looks the
// address up once with cudaGetSymbolAddress and caches it; make that first
// call before any stream capture.  All calls share the one array and it keeps
// the previous call's contents; the status word is cleared by every call, and
// the document starts are rewritten by every call that passes segment ids.
// Calls whose work overlaps on the GPU (for example on two streams) race on
// the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "hca_common.cuh"
#include "hca_internal.h"

namespace hca {
namespace {

// header (status word) + one int32 per (batch row, position)
constexpr long long kNoAllocMaxPositions = HCA_NOALLOC_MAX_POSITIONS;
constexpr size_t kNoAllocBytes = kHeaderBytes + kNoAllocMaxPositions * sizeof(int32_t);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_ptr(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace hca

using namespace hca;

extern "C" HCA_API int hca_attn_fwd_noalloc(const void *q, const void *kv, const void *ckv, const int32_t *seg,
                                            void *out, float *lse, int B, int H, int S, int D, int W, int m,
                                            float scale, int dtype, void *stream) {
  if ((long long)B * (long long)S > kNoAllocMaxPositions) return HCA_ERR_WORKSPACE;
  if (B < 0 || S < 0) return HCA_ERR_SHAPE;
  if ((long long)B * S == 0) {
    // nothing to compute; the ordinary entry point validates the rest
    return hca_attn_fwd(q, kv, ckv, seg, out, lse, B, H, S, D, W, m, scale, dtype, nullptr, 0, stream);
  }
  void *ws = nullptr;
  if (scratch_ptr(&ws) != cudaSuccess) return HCA_ERR_CUDA;
  return hca_attn_fwd(q, kv, ckv, seg, out, lse, B, H, S, D, W, m, scale, dtype, ws, kNoAllocBytes, stream);
}
