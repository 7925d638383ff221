// Declarations shared by the translation units of libvp (not part of the ABI).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace vp {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled, fetched from the driver through the runtime (the
// library does not link libcuda, so it loads on machines without a GPU).
EncodeTiledFn tensor_map_encoder();

// ---- bf16 tcgen05 path (ce_bf16.cu)
int lse_maxseg(int64_t V, int64_t Vs, int T);
int64_t lse_num_vtiles(int64_t V);
cudaError_t bf16_lse_stats(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                           int64_t Vs, float2* partial, int maxseg, float* zy, uint32_t* status,
                           cudaStream_t stream);
cudaError_t bf16_dz_chunk(const void* X, const void* W, const int64_t* targets, const float* lse, const float* g,
                          int64_t N, int64_t H, int64_t c0, int64_t Vc, void* dz, int64_t ldz, uint32_t* status,
                          cudaStream_t stream);
cudaError_t bf16_dx_chunk(const void* dz, int64_t ldz, const void* W, int64_t N, int64_t H, int64_t c0, int64_t Vc,
                          void* out, const float* partial, int mode, uint32_t* status, cudaStream_t stream);
cudaError_t bf16_dw_chunk(const void* dz, int64_t ldz, const void* X, int64_t N, int64_t H, int64_t c0, int64_t Vc,
                          float* dW, bool accumulate, uint32_t* status, cudaStream_t stream);
// Forward statistics plus p = exp(z - tile row max) in fp16 into P [N][ldp]
// and the tile row maxima into tmax [num_vtiles][N].
cudaError_t bf16_lse_stats_p(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                             int64_t Vs, float2* partial, int maxseg, float* zy, float* tmax, void* P, int64_t ldp,
                             uint32_t* status, cudaStream_t stream);
cudaError_t bf16_gemm_test(const void* A, const void* B, float* D, int64_t M, int64_t Ncols, int64_t K, int a_mn,
                           int b_mn, uint32_t* status, cudaStream_t stream);
// 1: tcgen05 GEMMs run as 2-SM CTA pairs (256 x 256 tiles); 0 (default): one SM per 128 x 256 tile.
void set_gemm_variant(int pair);
constexpr int kBf16TileV = 256;  // vocab width of one forward tile (statistics record granularity)

// ---- fp32 CUDA-core path (ce_simt.cu)
constexpr int kF32TileV = 64;
cudaError_t f32_lse_stats(const float* X, const float* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                          int64_t Vs, float2* partial, int maxseg, float* zy, cudaStream_t stream);
cudaError_t f32_dz_chunk(const float* X, const float* W, const int64_t* targets, const float* lse, const float* g,
                         int64_t N, int64_t H, int64_t c0, int64_t Vc, float* dz, int64_t ldz, cudaStream_t stream);
// C[M,N] (=|+=) sum_k A(m,k) B(k,n) with element strides.
cudaError_t f32_gemm(const float* A, int64_t sam, int64_t sak, const float* B, int64_t sbk, int64_t sbn, float* C,
                     int64_t ldc, int64_t M, int64_t Ncols, int64_t K, bool accumulate, cudaStream_t stream);
int f32_maxseg(int64_t V, int64_t Vs, int T);

// ---- merge / prep (merge.cu)
cudaError_t lse_merge(float2* partial, const float* zy, const int64_t* targets, int64_t N, int64_t V,
                      int64_t Vs, int T, int tile_v, int maxseg, int64_t ignore_index, float* loss, float* lse,
                      float* shard_stats, cudaStream_t stream);
// The same, for a block of N rows whose shard_stats rows sit in a [T][3][ss_ld] array.
// Both leave each shard's merged (m_t, S_t) in one of the records (scratch of the call).
cudaError_t lse_merge_ld(float2* partial, const float* zy, const int64_t* targets, int64_t N, int64_t V,
                         int64_t Vs, int T, int tile_v, int maxseg, int64_t ignore_index, float* loss, float* lse,
                         float* shard_stats, int64_t ss_ld, cudaStream_t stream);
// In place: P [N][ldp] fp16 probabilities relative to the tile row maxima
// tmax [ceil(V/256)][N] -> dZ bf16 = c p - g 1[j = y], c = g exp(tmax - lse).
cudaError_t dz_from_p(void* P, int64_t ldp, const float* tmax, const float* lse, const float* g,
                      const int64_t* targets, int64_t N, int64_t V, cudaStream_t stream);

cudaError_t loss_mean_and_bad(const float* loss, const int64_t* targets, int64_t N, int64_t V, int64_t ignore_index,
                              float* loss_mean, int32_t* n_bad, cudaStream_t stream);
cudaError_t upstream_scale(const int64_t* targets, const float* dloss, const float* dmean, int64_t N, int64_t V,
                           int64_t ignore_index,
                           float* g, cudaStream_t stream);

// ---- embedding (embed.cu)
cudaError_t embed_gather(const int64_t* ids, const void* W, void* out, int64_t N, int64_t H, int64_t V,
                         int64_t Vs, int T, int esize, cudaStream_t stream);

// ---- embedding backward (embed_bwd.cu)
size_t embed_bwd_workspace(int64_t N, int64_t H);
int embed_bwd_kernels(int64_t N);   // kernels one call launches (the dW memset not counted)
cudaError_t embed_bwd(const int64_t* ids, const void* dOut, float* dW, int64_t N, int64_t H, int64_t V, int esize,
                      bool accumulate, void* workspace, cudaStream_t stream);

}  // namespace vp
