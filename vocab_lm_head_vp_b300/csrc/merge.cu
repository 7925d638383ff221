// Per-token merge of the forward statistics and the small per-batch kernels.
//
// If a kernel earlier on the stream gave up a wait (a non-zero device status
// word), its records are incomplete: the merge then writes NaN to loss, lse
// and the shard statistics, so the failure shows in the outputs themselves.
//
// lse_merge: the on-device form of the pages' cross-shard reductions ("Vocab
// Parallelism" sec. 5.3.1; "Vocab parallelism: how to split embedding and LM
// head", figure 2 and key formulas).  A record (m, R) stands for a set of
// logits with maximum m and S = sum exp(z - m) = 1 + R: R sums every term
// but one maximal one, so the 1 is never added to a small R in fp32.  For
// token n, the per-tile records of shard t are merged into the shard's
// (m_t, R_t) (one thread per token and shard); the shards then merge into
// m = max_t m_t and R with S = 1 + R = sum_t S_t e^(m_t - m) (one thread per
// token, shards in order), and
//     loss = log1p(R) + (m - z_y)            (valid target; 0 otherwise),
//     lse  = m + log1p(R),
// the pages' l = log sum_j e^(z_j - m) - (z_y - m) as two non-negative
// terms: no cancellation when the target is the row's maximum and l << lse.
//
// loss_mean_and_bad: L = sum_n loss_n / max(1, N_valid) (sec. 5.3.3) and the
// count of targets that are neither ignore_index nor inside [0, V).
//
// upstream_scale: g_n = dloss_n (or dmean/max(1, N_valid), dmean = 1 when not
// given) on valid tokens, 0 on ignored ones -- the per-row factor of the logit
// gradient (sec. 5.3.2-5.3.3).
#include <cuda_runtime.h>

#include "vp_internal.h"

namespace vp {
namespace {

// (m, r) <- the merge of (m, r) and (m2, r2): the smaller maximum's whole set,
// 1 + r, is rescaled onto the larger one; the larger one's excluded term stays
// excluded.
__device__ __forceinline__ void merge_mr(float& m, float& r, float m2, float r2) {
  if (m2 > m) {
    r = r2 + (r + 1.f) * expf(m - m2);
    m = m2;
  } else {
    r += (r2 + 1.f) * expf(m2 - m);
  }
}

// Slot of shard t's first tile: where the shard's merged (m_t, R_t) is left.
__device__ __forceinline__ int64_t shard_slot(int t, int64_t Vs, int tile_v, int maxseg) {
  const int64_t nb = static_cast<int64_t>(t) * Vs / tile_v;
  const int k = t - static_cast<int>((nb * tile_v) / Vs);
  return nb * maxseg + k;
}

// One block per 32 tokens, 8 warps.  Step 1, warp w for shards w, w + 8, ...
// (lane = token): the shard's tile records, in tile order, into (m_t, R_t),
// written over the record of the shard's first tile (a record slot belongs to
// exactly one shard).  Step 2, warp 0 (one thread per token): the shards in
// order t = 0..T-1.
constexpr int kMergeBatch = 8;
constexpr int kMergeTokens = 32;
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(kMergeTokens * kMergeWarps)
    lse_merge_kernel(float2* __restrict__ partial, const float* __restrict__ zy, const int64_t* __restrict__ targets,
                     int64_t N, int64_t V, int64_t Vs, int T, int tile_v, int maxseg, int64_t ignore_index,
                     float* __restrict__ loss, float* __restrict__ lse, float* __restrict__ shard_stats,
                     int64_t ss_ld, const uint32_t* __restrict__ status) {
  const int lane = threadIdx.x % kMergeTokens, w = threadIdx.x / kMergeTokens;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * kMergeTokens + lane;
  if (n < N) {
    for (int t = w; t < T; t += kMergeWarps) {
      const int64_t a = static_cast<int64_t>(t) * Vs;
      const int64_t b = a + Vs;
      const int64_t nb0 = a / tile_v;
      // every record holds at least one logit: start from the shard's first one
      const float2 r0 = partial[(nb0 * maxseg + (t - static_cast<int>((nb0 * tile_v) / Vs))) * N + n];
      float mt = r0.x, rt = r0.y;
      const int64_t nb_last = (b - 1) / tile_v;
      int64_t nb = nb0 + 1;
      // the records of kMergeBatch tiles are loaded before any is merged, so that
      // their loads are in flight together; the merge order stays tile order
      for (; nb + kMergeBatch - 1 <= nb_last; nb += kMergeBatch) {
        float2 r[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const int k = t - static_cast<int>(((nb + u) * tile_v) / Vs);   // slot of shard t inside tile nb + u
          r[u] = partial[((nb + u) * maxseg + k) * N + n];
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) merge_mr(mt, rt, r[u].x, r[u].y);
      }
      for (; nb <= nb_last; ++nb) {
        const int k = t - static_cast<int>((nb * tile_v) / Vs);
        const float2 r = partial[(nb * maxseg + k) * N + n];
        merge_mr(mt, rt, r.x, r.y);
      }
      partial[shard_slot(t, Vs, tile_v, maxseg) * N + n] = make_float2(mt, rt);
    }
  }
  __syncthreads();   // every shard's (m_t, R_t) of the block's tokens is written
  if (w != 0 || n >= N) return;
  if (status && *status != 0u) {
    const float nan = __int_as_float(0x7fc00000);
    lse[n] = nan;
    loss[n] = nan;
    if (shard_stats)
      for (int64_t q = 0; q < 3 * static_cast<int64_t>(T); ++q) shard_stats[q * ss_ld + n] = nan;
    return;
  }
  const int64_t y = targets[n];
  const bool valid = y >= 0 && y < V && y != ignore_index;
  const float zyn = valid ? zy[n] : 0.f;
  float m = 0.f, r = 0.f;
  for (int t = 0; t < T; ++t) {
    const float2 rec = partial[shard_slot(t, Vs, tile_v, maxseg) * N + n];
    if (shard_stats) {
      const int64_t a = static_cast<int64_t>(t) * Vs;
      shard_stats[(static_cast<int64_t>(t) * 3 + 0) * ss_ld + n] = rec.x;
      shard_stats[(static_cast<int64_t>(t) * 3 + 1) * ss_ld + n] = 1.f + rec.y;   // S_t
      shard_stats[(static_cast<int64_t>(t) * 3 + 2) * ss_ld + n] = (valid && y >= a && y < a + Vs) ? zyn : 0.f;
    }
    if (t == 0) {
      m = rec.x;
      r = rec.y;
    } else {
      merge_mr(m, r, rec.x, rec.y);
    }
  }
  const float l1 = log1pf(r);
  lse[n] = m + l1;
  // z_y is one of the logits, so m - z_y >= 0: both terms are non-negative
  loss[n] = valid ? l1 + (m - zyn) : 0.f;
}

// One shard of a T-shard vocabulary computed by itself (a rank holding only
// its W_t): its tile records in order into (m_t, R_t), and its target logit
// z_y^(t) (0 when the target is ignored or in another shard).
__global__ void shard_stats_kernel(const float2* __restrict__ partial, const float* __restrict__ zy,
                                   const int64_t* __restrict__ targets, int64_t N, int64_t V, int64_t start,
                                   int64_t Vs, int64_t ntiles, int64_t ignore_index, float* __restrict__ stats,
                                   const uint32_t* __restrict__ status) {
  const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (n >= N) return;
  if (status && *status != 0u) {
    const float nan = __int_as_float(0x7fc00000);
    stats[n] = nan;
    stats[N + n] = nan;
    stats[2 * N + n] = nan;
    return;
  }
  const float2 r0 = partial[n];
  float m = r0.x, r = r0.y;
  int64_t nb = 1;
  for (; nb + kMergeBatch - 1 < ntiles; nb += kMergeBatch) {   // loads in flight together, merged in order
    float2 rec[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) rec[u] = partial[(nb + u) * N + n];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) merge_mr(m, r, rec[u].x, rec[u].y);
  }
  for (; nb < ntiles; ++nb) {
    const float2 rec = partial[nb * N + n];
    merge_mr(m, r, rec.x, rec.y);
  }
  const int64_t y = targets[n];
  const bool own = y >= start && y < start + Vs && y < V && y != ignore_index;
  stats[n] = m;
  stats[N + n] = r;
  stats[2 * N + n] = own ? zy[n] : 0.f;
}

// The merge of gathered shard statistics [T][3][N], shards in order: the
// pages' MAX of m_t, SUM of the rescaled local sums and SUM of z_y^(t).
__global__ void merge_shard_stats_kernel(const float* __restrict__ stats, const int64_t* __restrict__ targets,
                                         int64_t N, int64_t V, int T, int64_t ignore_index, float* __restrict__ loss,
                                         float* __restrict__ lse) {
  const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float m = stats[n], r = stats[N + n], z = 0.f + stats[2 * N + n];
  for (int t = 1; t < T; ++t) {
    const float* st = stats + static_cast<int64_t>(t) * 3 * N;
    merge_mr(m, r, st[n], st[N + n]);
    z += st[2 * N + n];
  }
  const int64_t y = targets[n];
  const bool valid = y >= 0 && y < V && y != ignore_index;
  const float l1 = log1pf(r);
  lse[n] = m + l1;
  loss[n] = valid ? l1 + (m - z) : 0.f;
}

constexpr int kRedThreads = 1024;

// One CTA: fixed-order (deterministic) sums over the batch.
__global__ void __launch_bounds__(kRedThreads) loss_mean_kernel(const float* __restrict__ loss,
                                                                const int64_t* __restrict__ targets, int64_t N,
                                                                int64_t V, int64_t ignore_index,
                                                                float* __restrict__ loss_mean,
                                                                int32_t* __restrict__ n_bad) {
  __shared__ double s_sum[kRedThreads];
  __shared__ int s_valid[kRedThreads];
  __shared__ int s_bad[kRedThreads];
  double sum = 0.0;
  int nv = 0, nbad = 0;
#pragma unroll 4
  for (int64_t n = threadIdx.x; n < N; n += kRedThreads) {
    const int64_t y = targets[n];
    const bool valid = y >= 0 && y < V && y != ignore_index;
    const bool in_range = y >= 0 && y < V;
    sum += valid ? static_cast<double>(loss[n]) : 0.0;
    nv += valid;
    nbad += (!in_range && y != ignore_index);
  }
  s_sum[threadIdx.x] = sum;
  s_valid[threadIdx.x] = nv;
  s_bad[threadIdx.x] = nbad;
  __syncthreads();
  for (int w = kRedThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s_sum[threadIdx.x] += s_sum[threadIdx.x + w];
      s_valid[threadIdx.x] += s_valid[threadIdx.x + w];
      s_bad[threadIdx.x] += s_bad[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int denom = s_valid[0] > 1 ? s_valid[0] : 1;
    if (loss_mean) *loss_mean = static_cast<float>(s_sum[0] / denom);
    if (n_bad) *n_bad = s_bad[0];
  }
}

__global__ void __launch_bounds__(kRedThreads) upstream_scale_kernel(const int64_t* __restrict__ targets,
                                                                     const float* __restrict__ dloss,
                                                                     const float* __restrict__ dmean, int64_t N,
                                                                     int64_t V, int64_t ignore_index,
                                                                     float* __restrict__ g) {
  __shared__ int s_valid[kRedThreads];
  int nv = 0;
#pragma unroll 4
  for (int64_t n = threadIdx.x; n < N; n += kRedThreads) {
    const int64_t y = targets[n];
    nv += (y >= 0 && y < V && y != ignore_index);
  }
  s_valid[threadIdx.x] = nv;
  __syncthreads();
  for (int w = kRedThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) s_valid[threadIdx.x] += s_valid[threadIdx.x + w];
    __syncthreads();
  }
  const float inv = (dmean ? *dmean : 1.0f) / static_cast<float>(s_valid[0] > 1 ? s_valid[0] : 1);
#pragma unroll 4
  for (int64_t n = threadIdx.x; n < N; n += kRedThreads) {
    const int64_t y = targets[n];
    const bool valid = y >= 0 && y < V && y != ignore_index;
    g[n] = valid ? (dloss ? dloss[n] : inv) : 0.f;
  }
}

}  // namespace

cudaError_t lse_merge_ld(float2* partial, const float* zy, const int64_t* targets, int64_t N, int64_t V,
                         int64_t Vs, int T, int tile_v, int maxseg, int64_t ignore_index, float* loss, float* lse,
                         float* shard_stats, int64_t ss_ld, const uint32_t* status, cudaStream_t stream) {
  // the records are scratch of this call: the shard step leaves each shard's merge in one of them
  const int64_t blocks = (N + kMergeTokens - 1) / kMergeTokens;
  lse_merge_kernel<<<static_cast<unsigned>(blocks), kMergeTokens * kMergeWarps, 0, stream>>>(
      partial, zy, targets, N, V, Vs, T, tile_v, maxseg, ignore_index, loss, lse, shard_stats, ss_ld, status);
  return cudaGetLastError();
}

cudaError_t lse_merge(float2* partial, const float* zy, const int64_t* targets, int64_t N, int64_t V,
                      int64_t Vs, int T, int tile_v, int maxseg, int64_t ignore_index, float* loss, float* lse,
                      float* shard_stats, const uint32_t* status, cudaStream_t stream) {
  return lse_merge_ld(partial, zy, targets, N, V, Vs, T, tile_v, maxseg, ignore_index, loss, lse, shard_stats, N,
                      status, stream);
}

cudaError_t shard_stats(const float2* partial, const float* zy, const int64_t* targets, int64_t N, int64_t V,
                        int64_t start, int64_t Vs, int64_t ntiles, int64_t ignore_index, float* stats,
                        const uint32_t* status, cudaStream_t stream) {
  const int threads = 256;
  shard_stats_kernel<<<static_cast<unsigned>((N + threads - 1) / threads), threads, 0, stream>>>(
      partial, zy, targets, N, V, start, Vs, ntiles, ignore_index, stats, status);
  return cudaGetLastError();
}

cudaError_t merge_shard_stats(const float* stats, const int64_t* targets, int64_t N, int64_t V, int T,
                              int64_t ignore_index, float* loss, float* lse, cudaStream_t stream) {
  const int threads = 256;
  merge_shard_stats_kernel<<<static_cast<unsigned>((N + threads - 1) / threads), threads, 0, stream>>>(
      stats, targets, N, V, T, ignore_index, loss, lse);
  return cudaGetLastError();
}

cudaError_t loss_mean_and_bad(const float* loss, const int64_t* targets, int64_t N, int64_t V, int64_t ignore_index,
                              float* loss_mean, int32_t* n_bad, cudaStream_t stream) {
  loss_mean_kernel<<<1, kRedThreads, 0, stream>>>(loss, targets, N, V, ignore_index, loss_mean, n_bad);
  return cudaGetLastError();
}

cudaError_t upstream_scale(const int64_t* targets, const float* dloss, const float* dmean, int64_t N, int64_t V,
                           int64_t ignore_index,
                           float* g, cudaStream_t stream) {
  upstream_scale_kernel<<<1, kRedThreads, 0, stream>>>(targets, dloss, dmean, N, V, ignore_index, g);
  return cudaGetLastError();
}

}  // namespace vp
