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
// device address is looked up once per device, with that device current.
struct DeviceScratch {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceScratch g_scratch[kNoAllocMaxDevices];

cudaError_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  DeviceScratch& d = g_scratch[dev];
  std::call_once(d.once, [&d] { d.err = cudaGetSymbolAddress(&d.ptr, g_noalloc_scratch); });
  if (d.err != cudaSuccess) return d.err;
  if (!d.ptr) return cudaErrorInvalidSymbol;
  *out = d.ptr;
  return cudaSuccess;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace vp

using namespace vp;

VP_EXPORT vp_status vp_lmhead_ce_fwd_noalloc(const void* X, const void* W, const int64_t* targets, int64_t N,
                                             int64_t H, int64_t V, int T, int64_t ignore_index, vp_dtype dtype,
                                             float* loss, float* lse, float* loss_mean, float* shard_stats,
                                             int32_t* n_bad, void* stream) {
  if (!X || !W || !targets || !loss || !lse) return VP_ERR_INVALID_ARG;
  if (dtype != VP_F32 && dtype != VP_BF16) return VP_ERR_INVALID_ARG;
  if (N <= 0 || H <= 0 || V <= 0 || T <= 0 || V % T != 0 || N >= (int64_t(1) << 31) || V >= (int64_t(1) << 31) ||
      H >= (int64_t(1) << 31))
    return VP_ERR_INVALID_ARG;
  const int es = dtype == VP_BF16 ? 2 : 4;
  const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(X) || !a16(W) || (H * es) % 16 != 0 || (reinterpret_cast<uintptr_t>(targets) & 7u) != 0)
    return VP_ERR_UNSUPPORTED;

  // Scratch layout: status word | (m, S) records per vocab tile and shard slot | z_y.
  const int64_t Vs = V / T;
  const int tile_v = dtype == VP_BF16 ? kBf16TileV : kF32TileV;
  const int maxseg = dtype == VP_BF16 ? lse_maxseg(V, Vs, T) : f32_maxseg(V, Vs, T);
  const int64_t ntiles = (V + tile_v - 1) / tile_v;
  const size_t off_partial = 256;
  const size_t off_zy = up256(off_partial + size_t(ntiles) * maxseg * size_t(N) * sizeof(float2));
  const size_t need = up256(off_zy + size_t(N) * sizeof(float));
  if (need > kNoAllocScratchBytes) return VP_ERR_WORKSPACE;   // beyond the fixed 32 MiB scratch
  if (dtype == VP_BF16 && !tensor_map_encoder()) return VP_ERR_CUDA;

  void* base = nullptr;
  if (scratch_on_current_device(&base) != cudaSuccess) return VP_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(base);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float2* partial = reinterpret_cast<float2*>(ws + off_partial);
  float* zy = reinterpret_cast<float*>(ws + off_zy);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The array keeps the previous call's contents: the status word must start at
  // zero; every record the merge reads is rewritten by this call's tiles.
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) {
    if (dtype == VP_BF16)
      e = bf16_lse_stats(X, W, targets, N, H, V, Vs, partial, maxseg, zy, status, s);
    else
      e = f32_lse_stats(static_cast<const float*>(X), static_cast<const float*>(W), targets, N, H, V, Vs, partial,
                        maxseg, zy, s);
  }
  if (e == cudaSuccess)
    e = lse_merge(partial, zy, targets, N, V, Vs, T, tile_v, maxseg, ignore_index, loss, lse, shard_stats, s);
  if (e == cudaSuccess && (loss_mean || n_bad))
    e = loss_mean_and_bad(loss, targets, N, V, ignore_index, loss_mean, n_bad, s);
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}
