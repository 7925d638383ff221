// fp32 path of the fused LM head + vocab-parallel cross-entropy on CUDA-core
// FMAs.  fp32 inputs are held to a 1e-5 relative loss tolerance, which TF32
// tensor cores cannot meet, so these kernels use plain fp32 arithmetic and
// the accurate expf/logf.  Same structure as the bf16 path: 64 x 64 logit
// tiles reduced to per-shard-segment (m, R) records (forward) or to dZ
// (backward), then plain GEMMs for dX and dW.
#include <cuda_runtime.h>

#include "vp_internal.h"

namespace vp {
namespace {

constexpr int kT = 64;    // tile rows / cols
constexpr int kK = 16;    // K step
constexpr int kThr = 256; // 16 x 16 threads, 4 x 4 outputs each

// acc[i][j] = sum_k A(r0 + ty*4 + i, k) * B(k, c0 + tx*4 + j) with
// A(m,k) = A[m*sam + k*sak] (m < M), B(k,n) = B[k*sbk + n*sbn] (n < Ncols).
__device__ __forceinline__ void tile_mma(const float* __restrict__ A, int64_t sam, int64_t sak, int64_t M,
                                         const float* __restrict__ B, int64_t sbk, int64_t sbn, int64_t Ncols,
                                         int64_t K, int64_t r0, int64_t c0, float (&acc)[4][4],
                                         float (*As)[kT + 4], float (*Bs)[kT + 4]) {
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int64_t k0 = 0; k0 < K; k0 += kK) {
    // 64 x 16 elements of A and 16 x 64 of B; 4 per thread each
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = tid + q * kThr;       // 0..1023
      const int mm = e / kK, kk = e % kK; // A: row-of-tile, k
      const int64_t gm = r0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < K) ? A[gm * sam + gk * sak] : 0.f;
      const int nn = e % kT, kb = e / kT; // B: k, col-of-tile
      const int64_t gn = c0 + nn, gkb = k0 + kb;
      Bs[kb][nn] = (gn < Ncols && gkb < K) ? B[gkb * sbk + gn * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
}

// Forward: Z tile = X[n0:n0+64] W[v0:v0+64]^T -> per-row shard-segment records
// (m, R): the segment's maximum and the sum of exp(z - m) over its logits
// except one maximal one (S = 1 + R).
__global__ void __launch_bounds__(kThr) f32_lse_kernel(const float* __restrict__ X, const float* __restrict__ W,
                                                       const int64_t* __restrict__ targets, int64_t N, int64_t H,
                                                       int64_t V, int64_t Vs, float2* __restrict__ partial,
                                                       int maxseg, float* __restrict__ zy, int64_t y_off) {
  __shared__ float As[kK][kT + 4];
  __shared__ float Bs[kK][kT + 4];
  __shared__ float Zs[kT][kT + 1];
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kT;
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kT;
  float acc[4][4];
  // B(k, v) = W[v*H + k]
  tile_mma(X, H, 1, N, W, 1, H, V, H, n0, v0, acc, As, Bs);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Zs[ty * 4 + i][tx * 4 + j] = acc[i][j];
  __syncthreads();
  if (threadIdx.x >= kT) return;
  const int r = threadIdx.x;
  const int64_t n = n0 + r;
  if (n >= N) return;
  const int64_t vend = min(v0 + kT, V);
  const int64_t y = targets[n];
  int64_t t = v0 / Vs;
  int64_t seg_end = min((t + 1) * Vs, vend);
  int k = 0;
  float m = -INFINITY, s = 0.f;
  float2* rec = partial + (static_cast<int64_t>(blockIdx.x) * maxseg) * N + n;
  for (int64_t col = v0; col < vend; ++col) {
    if (col == seg_end) {
      rec[static_cast<int64_t>(k) * N] = make_float2(m, s);
      ++k;
      ++t;
      seg_end = min((t + 1) * Vs, vend);
      m = -INFINITY;
      s = 0.f;
    }
    const float z = Zs[r][col - v0];
    if (z > m) {
      s = (s + 1.f) * expf(m - z);   // the old maximum joins the sum (expf(-inf) = 0 at the start)
      m = z;
    } else {
      s += expf(z - m);              // a tie adds exp(0) = 1
    }
    if (col + y_off == y) zy[n] = z;
  }
  rec[static_cast<int64_t>(k) * N] = make_float2(m, s);
}

// Backward: dZ[n, c] = g_n (exp(z - lse_n) - 1[c0 + c = y_n]) for chunk columns c < Vc.
__global__ void __launch_bounds__(kThr) f32_dz_kernel(const float* __restrict__ X, const float* __restrict__ W,
                                                      const int64_t* __restrict__ targets,
                                                      const float* __restrict__ lse, const float* __restrict__ g,
                                                      int64_t N, int64_t H, int64_t c0, int64_t Vc,
                                                      float* __restrict__ dz, int64_t ldz, int64_t y_off) {
  __shared__ float As[kK][kT + 4];
  __shared__ float Bs[kK][kT + 4];
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kT;
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kT;  // chunk-local
  float acc[4][4];
  tile_mma(X, H, 1, N, W + c0 * H, 1, H, Vc, H, n0, v0, acc, As, Bs);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t n = n0 + ty * 4 + i;
    if (n >= N) continue;
    const float gn = g[n], ln = lse[n];
    const int64_t yl = targets[n] - y_off - c0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t c = v0 + tx * 4 + j;
      if (c >= Vc) continue;
      float d = gn * expf(acc[i][j] - ln);
      if (c == yl) d -= gn;
      dz[n * ldz + c] = d;
    }
  }
}

__global__ void __launch_bounds__(kThr) f32_gemm_kernel(const float* __restrict__ A, int64_t sam, int64_t sak,
                                                        const float* __restrict__ B, int64_t sbk, int64_t sbn,
                                                        float* __restrict__ C, int64_t ldc, int64_t M, int64_t Ncols,
                                                        int64_t K, int accumulate) {
  __shared__ float As[kK][kT + 4];
  __shared__ float Bs[kK][kT + 4];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kT;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kT;
  float acc[4][4];
  tile_mma(A, sam, sak, M, B, sbk, sbn, Ncols, K, r0, c0, acc, As, Bs);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = r0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = c0 + tx * 4 + j;
      if (n >= Ncols) continue;
      float* c = C + m * ldc + n;
      *c = accumulate ? *c + acc[i][j] : acc[i][j];
    }
  }
}

dim3 tiles(int64_t rows, int64_t cols) {
  return dim3(static_cast<unsigned>((cols + kT - 1) / kT), static_cast<unsigned>((rows + kT - 1) / kT));
}

}  // namespace

int f32_maxseg(int64_t V, int64_t Vs, int T) {
  (void)V;
  int64_t m = (kT - 1) / Vs + 2;
  if (m > T) m = T;
  return static_cast<int>(m);
}

cudaError_t f32_lse_stats(const float* X, const float* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                          int64_t Vs, float2* partial, int maxseg, float* zy, cudaStream_t stream, int64_t y_off) {
  f32_lse_kernel<<<tiles(N, V), kThr, 0, stream>>>(X, W, targets, N, H, V, Vs, partial, maxseg, zy, y_off);
  return cudaGetLastError();
}

cudaError_t f32_dz_chunk(const float* X, const float* W, const int64_t* targets, const float* lse, const float* g,
                         int64_t N, int64_t H, int64_t c0, int64_t Vc, float* dz, int64_t ldz, cudaStream_t stream,
                         int64_t y_off) {
  f32_dz_kernel<<<tiles(N, Vc), kThr, 0, stream>>>(X, W, targets, lse, g, N, H, c0, Vc, dz, ldz, y_off);
  return cudaGetLastError();
}

cudaError_t f32_gemm(const float* A, int64_t sam, int64_t sak, const float* B, int64_t sbk, int64_t sbn, float* C,
                     int64_t ldc, int64_t M, int64_t Ncols, int64_t K, bool accumulate, cudaStream_t stream) {
  f32_gemm_kernel<<<tiles(M, Ncols), kThr, 0, stream>>>(A, sam, sak, B, sbk, sbn, C, ldc, M, Ncols, K,
                                                         accumulate ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace vp
