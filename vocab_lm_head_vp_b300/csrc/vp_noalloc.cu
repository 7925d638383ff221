// vp_lmhead_ce_fwd_noalloc: the fused LM head + cross-entropy forward for
// callers that have no way to hand the library a device workspace.
//
// Some callers cannot allocate device memory at all: a plugin whose host
// passes it only its input and output buffers and offers no allocator, or a
// latency-bound loop that must never call cudaMalloc (it can synchronise the
// whole device and takes unbounded time).  This entry point needs nothing but
// the inputs and outputs: its scratch (the per-tile statistics records, the
// target logits and the device status word) lives in one file-scope device
// array of fixed size that every GPU holds from the moment it loads this
// library until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/vp.h"
#include "vp_internal.h"

#define VP_EXPORT extern "C" __attribute__((visibility("default")))

namespace vp {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB per GPU
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// In host code `g_noalloc_scratch` only names a host-side stand-in; the
// device address is looked up with the device current, the first time a call
// runs on that device, and kept for later calls on it.  A failed lookup is not
// kept: the next call tries again.
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kNoAllocMaxDevices] = {};

cudaError_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace vp

using namespace vp;

VP_EXPORT vp_status vp_lmhead_ce_fwd_noalloc(const void* X, const void* W, const int64_t* targets, int64_t N,
                                             int64_t H, int64_t V, int T, int64_t ignore_index, vp_dtype dtype,
                                             float* loss, float* lse, float* loss_mean, float* shard_stats,
                                             int32_t* n_bad, void* stream) {
  if (!loss || !lse) return VP_ERR_INVALID_ARG;
  const vp_status st = check_inputs(X, W, targets, N, H, V, T, dtype);
  if (st != VP_OK) return st;
  // the same scratch layout as vp_lmhead_ce_fwd's workspace
  const FwdLayout L = fwd_layout(N, V, T, dtype);
  if (L.total > kNoAllocScratchBytes) return VP_ERR_WORKSPACE;   // beyond the fixed 32 MiB scratch
  if (dtype == VP_BF16 && !tensor_map_encoder()) return VP_ERR_CUDA;

  void* base = nullptr;
  if (scratch_on_current_device(&base) != cudaSuccess) return VP_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(base);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float2* partial = reinterpret_cast<float2*>(ws + L.off_partial);
  float* zy = reinterpret_cast<float*>(ws + L.off_zy);
  const int64_t Vs = V / T;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The array keeps the previous call's contents: the status word must start at
  // zero; every record the merge reads is rewritten by this call's tiles.  The
  // status word cannot be read through vp_read_device_status; a kernel that
  // gives up a wait makes the merge write NaN to loss and lse instead.
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) {
    if (dtype == VP_BF16)
      e = bf16_lse_stats(X, W, targets, N, H, V, Vs, partial, L.maxseg, zy, status, s);
    else
      e = f32_lse_stats(static_cast<const float*>(X), static_cast<const float*>(W), targets, N, H, V, Vs, partial,
                        L.maxseg, zy, s);
  }
  if (e == cudaSuccess)
    e = lse_merge(partial, zy, targets, N, V, Vs, T, L.tile_v, L.maxseg, ignore_index, loss, lse, shard_stats,
                  status, s);
  if (e == cudaSuccess && (loss_mean || n_bad))
    e = loss_mean_and_bad(loss, targets, N, V, ignore_index, loss_mean, n_bad, s);
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}
