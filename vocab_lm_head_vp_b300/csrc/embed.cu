// Vocab-parallel embedding gather ("Vocab Parallelism" sec. 5.2.1; "Vocab
// parallelism: how to split embedding and LM head", figure 1).
//
// Shard t answers an id only inside [t*Vs, (t+1)*Vs): it reads local row
// id - t*Vs of its slice W_t = W[t*Vs : (t+1)*Vs] and every other shard
// contributes a zero row.  Summing the T shard outputs therefore equals
// +0.0 + (the owner's row), so the kernel reads only the owning shard's row
// (none for an out-of-range id) and adds the zero rows implicitly: the one
// visible effect of the sum, -0.0 -> +0.0, is applied bit-wise.
//
// HBM-bound copy: 16-byte vector loads and stores, four in flight per thread,
// consecutive threads on consecutive 16-byte pieces of a row.
#include <cuda_runtime.h>

#include "vp_internal.h"

namespace vp {
namespace {

constexpr int kEmbThreads = 256;
constexpr int kEmbUnroll = 4;

// +0.0 + x for every element of a 16-byte vector, as bit operations.
__device__ __forceinline__ uint32_t canon_bf16x2(uint32_t w) { return w & ~__vcmpeq2(w, 0x80008000u); }
__device__ __forceinline__ uint32_t canon_f32(uint32_t w) { return w == 0x80000000u ? 0u : w; }

template <int ESIZE>
__global__ void __launch_bounds__(kEmbThreads) embed_gather_kernel(const int64_t* __restrict__ ids,
                                                                   const uint4* __restrict__ W,
                                                                   uint4* __restrict__ out, int64_t N,
                                                                   int64_t rowvec, int64_t V, int64_t Vs) {
  const int64_t total = N * rowvec;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * (kEmbThreads * kEmbUnroll) + threadIdx.x;
  uint4 v[kEmbUnroll];
#pragma unroll
  for (int u = 0; u < kEmbUnroll; ++u) {
    const int64_t idx = base + u * kEmbThreads;
    v[u] = make_uint4(0u, 0u, 0u, 0u);
    if (idx < total) {
      const int64_t n = idx / rowvec;
      const int64_t piece = idx - n * rowvec;
      const int64_t id = __ldg(ids + n);
      if (id >= 0 && id < V) {
        const int64_t t = id / Vs;            // owning shard
        const int64_t local = id - t * Vs;    // row inside W_t
        v[u] = __ldg(W + (t * Vs + local) * rowvec + piece);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kEmbUnroll; ++u) {
    const int64_t idx = base + u * kEmbThreads;
    if (idx < total) {
      uint4 w = v[u];
      if (ESIZE == 2) {
        w.x = canon_bf16x2(w.x);
        w.y = canon_bf16x2(w.y);
        w.z = canon_bf16x2(w.z);
        w.w = canon_bf16x2(w.w);
      } else {
        w.x = canon_f32(w.x);
        w.y = canon_f32(w.y);
        w.z = canon_f32(w.z);
        w.w = canon_f32(w.w);
      }
      out[idx] = w;
    }
  }
}

}  // namespace

cudaError_t embed_gather(const int64_t* ids, const void* W, void* out, int64_t N, int64_t H, int64_t V, int64_t Vs,
                         int /*T*/, int esize, cudaStream_t stream) {
  const int64_t rowvec = H * esize / 16;
  const int64_t total = N * rowvec;
  const int64_t per_block = kEmbThreads * kEmbUnroll;
  const int64_t blocks = (total + per_block - 1) / per_block;
  if (blocks == 0) return cudaSuccess;
  if (esize == 2)
    embed_gather_kernel<2><<<static_cast<unsigned>(blocks), kEmbThreads, 0, stream>>>(
        ids, static_cast<const uint4*>(W), static_cast<uint4*>(out), N, rowvec, V, Vs);
  else
    embed_gather_kernel<4><<<static_cast<unsigned>(blocks), kEmbThreads, 0, stream>>>(
        ids, static_cast<const uint4*>(W), static_cast<uint4*>(out), N, rowvec, V, Vs);
  return cudaGetLastError();
}

}  // namespace vp
