// Saved-probability backward step of the fused LM head + cross-entropy
// ("Vocab Parallelism" sec. 5.3.2: the logit gradient of shard t is the local
// softmax minus the local one-hot, dL/dz_j = g (p_j - 1[j = y]), with no
// communication; sec. 5.3.3: ignored rows get g = 0).
//
// The fused forward leaves, for token row n and 256-wide vocab tile k,
//     P[n, j] = fp16(exp(z_nj - tmax[k][n]))        (j inside tile k)
// where tmax[k][n] is the row's maximum over that tile.  Once the merge has
// produced lse_n, the softmax is p_nj = P[n, j] * exp(tmax[k][n] - lse_n), so
//     dZ[n, j] = bf16( c_nk * P[n, j] - g_n 1[j = y_n] ),  c_nk = g_n exp(tmax[k][n] - lse_n).
//
// tile_scale turns tmax into c in place (one multiply per element is left for
// the pass over P); dz_from_p then writes dZ over P in place (both elements
// are 2 bytes).
//
// HBM-bound elementwise pass: 16-byte vectors (8 elements, all inside one
// tile), consecutive threads on consecutive vectors of a row, kDzVecs vectors
// in flight per thread; a warp covers exactly one tile, so its tmax read is a
// broadcast.  Rows with g_n = 0 are written as zeros without being read.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "vp_internal.h"

namespace vp {
namespace {

constexpr int kDzThreads = 256;
// Two vectors per thread and 8 blocks per SM (32 registers, full occupancy)
// measured fastest on B300 at V=128256 (1.53 ms against 2.38 ms for 4 vectors
// per thread at 47 registers, same box).
#ifndef VP_DZ_VECS
#define VP_DZ_VECS 2
#endif
#ifndef VP_DZ_MIN_BLOCKS
#define VP_DZ_MIN_BLOCKS 8
#endif
constexpr int kDzVecs = VP_DZ_VECS;    // vectors per thread, kDzThreads apart
constexpr int kDzVecsPerTile = kBf16TileV / 8;
static_assert(kDzThreads % kDzVecsPerTile == 0, "a warp's vectors must stay inside one tile");

__device__ __forceinline__ uint32_t scale_pair(uint32_t h2, float c, int j0, int64_t yl, float g) {
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  float2 f = __half22float2(h);
  float a = c * f.x, b = c * f.y;
  if (yl == j0) a -= g;
  if (yl == j0 + 1) b -= g;
  __nv_bfloat162 o = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&o);
}

__global__ void tile_scale_kernel(float* __restrict__ tmax_c, const float* __restrict__ lse,
                                  const float* __restrict__ g, int64_t N, int64_t ntiles) {
  const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const float gn = g[n], ln = lse[n];
  for (int64_t k = blockIdx.y; k < ntiles; k += gridDim.y) {
    float* x = tmax_c + k * N + n;
    *x = gn * expf(*x - ln);
  }
}

__global__ void __launch_bounds__(kDzThreads, VP_DZ_MIN_BLOCKS)
    dz_from_p_kernel(uint4* __restrict__ buf, int64_t ldv, int64_t nvec, const float* __restrict__ cscale,
                     const float* __restrict__ g, const int64_t* __restrict__ targets, int64_t N) {
  const int64_t base = static_cast<int64_t>(blockIdx.x) * (kDzThreads * kDzVecs) + threadIdx.x;
  for (int64_t n = blockIdx.y; n < N; n += gridDim.y) {
    const float gn = g[n];
    uint4* row = buf + n * ldv;
    if (gn == 0.f) {
#pragma unroll
      for (int u = 0; u < kDzVecs; ++u) {
        const int64_t idx = base + u * kDzThreads;
        if (idx < nvec) row[idx] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    const int64_t y = targets[n];
    uint4 v[kDzVecs];
#pragma unroll
    for (int u = 0; u < kDzVecs; ++u) {
      const int64_t idx = base + u * kDzThreads;
      if (idx < nvec) v[u] = row[idx];
    }
#pragma unroll
    for (int u = 0; u < kDzVecs; ++u) {
      const int64_t idx = base + u * kDzThreads;
      if (idx < nvec) {
        const int64_t j0 = idx * 8;
        const float c = cscale[(j0 / kBf16TileV) * N + n];
        const int64_t yl = y - j0;   // target position inside this vector, if 0 <= yl < 8
        uint4 o;
        o.x = scale_pair(v[u].x, c, 0, yl, gn);
        o.y = scale_pair(v[u].y, c, 2, yl, gn);
        o.z = scale_pair(v[u].z, c, 4, yl, gn);
        o.w = scale_pair(v[u].w, c, 6, yl, gn);
        row[idx] = o;
      }
    }
  }
}

}  // namespace

cudaError_t tile_scale(float* tmax_c, const float* lse, const float* g, int64_t N, int64_t V, cudaStream_t stream) {
  if (N <= 0 || V <= 0) return cudaSuccess;
  const int64_t ntiles = (V + kBf16TileV - 1) / kBf16TileV;
  const dim3 grid(static_cast<unsigned>((N + 255) / 256), static_cast<unsigned>(ntiles < 65535 ? ntiles : 65535));
  tile_scale_kernel<<<grid, 256, 0, stream>>>(tmax_c, lse, g, N, ntiles);
  return cudaGetLastError();
}

cudaError_t dz_from_p(void* P, int64_t ldp, const float* cscale, const float* g, const int64_t* targets, int64_t N,
                      int64_t V, cudaStream_t stream) {
  if (N <= 0 || V <= 0) return cudaSuccess;
  const int64_t nvec = (V + 7) / 8;   // vectors holding columns < V (the last may run into the row padding)
  const int64_t per_block = kDzThreads * kDzVecs;
  const dim3 grid(static_cast<unsigned>((nvec + per_block - 1) / per_block),
                  static_cast<unsigned>(N < 65535 ? N : 65535));
  dz_from_p_kernel<<<grid, kDzThreads, 0, stream>>>(static_cast<uint4*>(P), ldp / 8, nvec, cscale, g, targets, N);
  return cudaGetLastError();
}

}  // namespace vp
