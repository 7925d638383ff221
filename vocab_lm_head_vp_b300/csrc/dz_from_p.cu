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
// dz_from_p writes dZ over P in place (both elements are 2 bytes).
//
// HBM-bound elementwise pass: 16-byte vectors (8 elements, all inside one
// tile), consecutive threads on consecutive vectors of a row, kDzVecs vectors
// in flight per thread.  A warp covers exactly one tile of one row, so c_nk
// costs a broadcast load of tmax and one hardware exp2 per lane, next to 512
// bytes of P moved per warp.  Rows with g_n = 0 are written as zeros without being read.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
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
constexpr float kLog2e = 1.4426950408889634f;   // exp(x) = 2^(x log2 e)
static_assert(kDzThreads % kDzVecsPerTile == 0, "a warp's vectors must stay inside one tile");

// dZ for one 16-byte vector of P: 8 products c p, then, only in the one vector
// per row that holds the target column (0 <= yl < 8), its -g.
__device__ __forceinline__ uint4 scale_vec(uint4 v, float c, int64_t yl, float g) {
  float f[8];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h2 = w[q];
    const float2 t = __half22float2(*reinterpret_cast<__half2*>(&h2));
    f[2 * q] = c * t.x;
    f[2 * q + 1] = c * t.y;
  }
  if (static_cast<uint64_t>(yl) < 8u) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q == yl) f[q] -= g;
  }
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * q], f[2 * q + 1]);
    o[q] = *reinterpret_cast<uint32_t*>(&b);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Vector indices within a row fit in 32 bits (the launcher checks it).
__global__ void __launch_bounds__(kDzThreads, VP_DZ_MIN_BLOCKS)
    dz_from_p_kernel(uint4* __restrict__ buf, int64_t ldv, int nvec, const float* __restrict__ tmax,
                     const float* __restrict__ lse, const float* __restrict__ g,
                     const int64_t* __restrict__ targets, int64_t N) {
  const int base = static_cast<int>(blockIdx.x) * (kDzThreads * kDzVecs) + static_cast<int>(threadIdx.x);
  for (int64_t n = blockIdx.y; n < N; n += gridDim.y) {
    const float gn = g[n];
    uint4* row = buf + n * ldv;
    if (gn == 0.f) {
#pragma unroll
      for (int u = 0; u < kDzVecs; ++u) {
        const int idx = base + u * kDzThreads;
        if (idx < nvec) row[idx] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    const float ln = lse[n];
    const int64_t y = targets[n];
    uint4 v[kDzVecs];
#pragma unroll
    for (int u = 0; u < kDzVecs; ++u) {
      const int idx = base + u * kDzThreads;
      if (idx < nvec) v[u] = row[idx];
    }
#pragma unroll
    for (int u = 0; u < kDzVecs; ++u) {
      const int idx = base + u * kDzThreads;
      if (idx < nvec) {
        // tile of this vector: kDzVecsPerTile vectors per tile.  One MUFU op for
        // exp: its relative error (~2^-22) is far below the bf16 rounding of dZ.
        const float t = tmax[static_cast<int64_t>(static_cast<unsigned>(idx) / kDzVecsPerTile) * N + n];
        const float c = gn * ex2_approx((t - ln) * kLog2e);
        row[idx] = scale_vec(v[u], c, y - static_cast<int64_t>(idx) * 8, gn);
      }
    }
  }
}

}  // namespace

cudaError_t dz_from_p(void* P, int64_t ldp, const float* tmax, const float* lse, const float* g,
                      const int64_t* targets, int64_t N, int64_t V, cudaStream_t stream) {
  if (N <= 0 || V <= 0) return cudaSuccess;
  const int64_t nvec = (V + 7) / 8;   // vectors holding columns < V (the last may run into the row padding)
  const int64_t per_block = kDzThreads * kDzVecs;
  if (nvec > INT32_MAX - per_block) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>((nvec + per_block - 1) / per_block),
                  static_cast<unsigned>(N < 65535 ? N : 65535));
  dz_from_p_kernel<<<grid, kDzThreads, 0, stream>>>(static_cast<uint4*>(P), ldp / 8, static_cast<int>(nvec), tmax, lse,
                                                     g, targets, N);
  return cudaGetLastError();
}

}  // namespace vp
