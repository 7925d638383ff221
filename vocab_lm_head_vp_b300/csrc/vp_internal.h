// Declarations shared by the translation units of libvp (not part of the ABI).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/vp.h"

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
// y_off: the vocab id of W's first row when W holds one shard of a larger
// vocabulary (targets are then ids of the whole vocabulary); 0 otherwise.
cudaError_t bf16_lse_stats(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                           int64_t Vs, float2* partial, int maxseg, float* zy, uint32_t* status,
                           cudaStream_t stream, int64_t y_off = 0);
cudaError_t bf16_dz_chunk(const void* X, const void* W, const int64_t* targets, const float* lse, const float* g,
                          int64_t N, int64_t H, int64_t c0, int64_t Vc, void* dz, int64_t ldz, uint32_t* status,
                          cudaStream_t stream, int64_t y_off = 0);
// sk_ws: sk_workspace_bytes() of fp32 scratch for stream-K partial tiles (the
// launch splits the (tile, k-block) iterations evenly over the SMs when its
// tiles do not fill whole waves); nullptr: whole tiles only.
cudaError_t bf16_dx_chunk(const void* dz, int64_t ldz, const void* W, int64_t N, int64_t H, int64_t c0, int64_t Vc,
                          void* out, const float* partial, int mode, uint32_t* status, cudaStream_t stream,
                          float* sk_ws = nullptr, int* kernels = nullptr);
size_t sk_workspace_bytes();
// How bf16_dx_chunk runs a dX GEMM over `rows` token rows: tile rows (128 or
// 256), whether stream-K, and the relative time (waves of 128 x 256 tiles).
struct DxPlan {
  int rows;
  bool streamk;
  double cost;
};
DxPlan dx_plan(int64_t rows, int64_t H);
// The same plan for a grid of G persistent CTAs (dx_plan: the device's SM count).
DxPlan dx_plan_on(int64_t rows, int64_t H, int64_t G);
// dW through X^T (A K-major): Xt = X^T [H][ldxt] bf16 (transpose_bf16 of X).
// cudaErrorNotSupported under GEMM form 2 (callers then use bf16_dw_chunk).
cudaError_t bf16_dwt_chunk(const void* Xt, int64_t ldxt, const void* dz, int64_t ldz, int64_t N, int64_t H,
                           int64_t c0, int64_t Vc, float* dW, bool accumulate, uint32_t* status, cudaStream_t stream);
// out[c][r] = in[r][c], bf16, cols a multiple of 8.
cudaError_t transpose_bf16(const void* in, int64_t rows, int64_t cols, int64_t ld_in, void* out, int64_t ld_out,
                           cudaStream_t stream);
// Whether the dW GEMMs take the X^T form (GEMM forms 0 and 1).
bool dw_through_xt();
cudaError_t bf16_dw_chunk(const void* dz, int64_t ldz, const void* X, int64_t N, int64_t H, int64_t c0, int64_t Vc,
                          float* dW, bool accumulate, uint32_t* status, cudaStream_t stream);
// Forward statistics plus p = exp(z - tile row max) in fp16 into P [N][ldp]
// and the tile row maxima into tmax [num_vtiles][N].
cudaError_t bf16_lse_stats_p(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                             int64_t Vs, float2* partial, int maxseg, float* zy, float* tmax, void* P, int64_t ldp,
                             uint32_t* status, cudaStream_t stream);
cudaError_t bf16_gemm_test(const void* A, const void* B, float* D, int64_t M, int64_t Ncols, int64_t K, int a_mn,
                           int b_mn, uint32_t* status, cudaStream_t stream);
// 0 (default): one SM per tile, dX in 256 x 256 tiles, the other GEMMs in
// 128 x 256; 1: 2-SM CTA pairs (256 x 256 tiles); 2: one SM per 128 x 256 tile.
void set_gemm_variant(int variant);
// Later one-SM GEMM launches: hold = 1 (the TMA producer issues no load) or
// 2 (the MMA issuer issues no MMA), 0 = none; every mbarrier wait gives up
// after wait_ns (0 = the default limit).
void set_wait_fault(int hold, uint64_t wait_ns);
constexpr int kBf16TileV = 256;  // vocab width of one forward tile (statistics record granularity)

// ---- fp32 CUDA-core path (ce_simt.cu)
constexpr int kF32TileV = 64;
cudaError_t f32_lse_stats(const float* X, const float* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                          int64_t Vs, float2* partial, int maxseg, float* zy, cudaStream_t stream, int64_t y_off = 0);
cudaError_t f32_dz_chunk(const float* X, const float* W, const int64_t* targets, const float* lse, const float* g,
                         int64_t N, int64_t H, int64_t c0, int64_t Vc, float* dz, int64_t ldz, cudaStream_t stream,
                         int64_t y_off = 0);
// C[M,N] (=|+=) sum_k A(m,k) B(k,n) with element strides.
cudaError_t f32_gemm(const float* A, int64_t sam, int64_t sak, const float* B, int64_t sbk, int64_t sbn, float* C,
                     int64_t ldc, int64_t M, int64_t Ncols, int64_t K, bool accumulate, cudaStream_t stream);
int f32_maxseg(int64_t V, int64_t Vs, int T);

// ---- merge / prep (merge.cu)
// Records (m, R): maximum and sum of exp(z - m) without one maximal term.
// A non-zero *status (a kernel gave up a wait) makes loss, lse and shard_stats NaN.
cudaError_t lse_merge(float2* partial, const float* zy, const int64_t* targets, int64_t N, int64_t V,
                      int64_t Vs, int T, int tile_v, int maxseg, int64_t ignore_index, float* loss, float* lse,
                      float* shard_stats, const uint32_t* status, cudaStream_t stream);
// The same, for a block of N rows whose shard_stats rows sit in a [T][3][ss_ld] array.
// Both leave each shard's merged (m_t, R_t) in one of the records (scratch of the call).
cudaError_t lse_merge_ld(float2* partial, const float* zy, const int64_t* targets, int64_t N, int64_t V,
                         int64_t Vs, int T, int tile_v, int maxseg, int64_t ignore_index, float* loss, float* lse,
                         float* shard_stats, int64_t ss_ld, const uint32_t* status, cudaStream_t stream);
// In place: P [N][ldp] fp16 probabilities relative to the tile row maxima
// tmax [ceil(V/256)][N] -> dZ bf16 = c p - g 1[j = y], c = g exp(tmax - lse).
cudaError_t dz_from_p(void* P, int64_t ldp, const float* tmax, const float* lse, const float* g,
                      const int64_t* targets, int64_t N, int64_t V, cudaStream_t stream);

// One vocab shard's statistics [3][N] = (m_t, R_t, z_y^(t)) from the records
// of a call over that shard alone (one record per 256- or 64-wide tile,
// `ntiles` of them); targets are ids of the whole vocabulary [0, V), the
// shard holds [start, start + Vs).
cudaError_t shard_stats(const float2* partial, const float* zy, const int64_t* targets, int64_t N, int64_t V,
                        int64_t start, int64_t Vs, int64_t ntiles, int64_t ignore_index, float* stats,
                        const uint32_t* status, cudaStream_t stream);
// The merge of T shards' statistics [T][3][N] (gathered from the shards'
// calls) into loss and lse.
cudaError_t merge_shard_stats(const float* stats, const int64_t* targets, int64_t N, int64_t V, int T,
                              int64_t ignore_index, float* loss, float* lse, cudaStream_t stream);

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
int embed_bwd_sort_kernels(int64_t N);   // kernels embed_bwd_sort launches
// Step 1, ids only: the tokens' (id, n) keys sorted into the workspace.
cudaError_t embed_bwd_sort(const int64_t* ids, int64_t N, int64_t V, void* workspace, cudaStream_t stream);
// Steps 2-3 (two kernels, after a dW memset when not accumulating): the sums
// over the keys embed_bwd_sort left in the same workspace.
cudaError_t embed_bwd_sums(const void* dOut, float* dW, int64_t N, int64_t H, int64_t V, int esize, bool accumulate,
                           void* workspace, cudaStream_t stream);

// ---- argument checks and the forward workspace layout (vp_api.cu, vp_noalloc.cu)
constexpr size_t kAlign = 256;
constexpr size_t kHeader = 256;  // device status word + reserved

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int esize_of(vp_dtype dt) { return dt == VP_BF16 ? 2 : 4; }
inline bool dtype_ok(int dt) { return dt == VP_F32 || dt == VP_BF16; }

inline bool shape_ok(int64_t N, int64_t H, int64_t V, int T) {
  return N > 0 && H > 0 && V > 0 && T > 0 && V % T == 0 && N < (int64_t(1) << 31) && V < (int64_t(1) << 31) &&
         H < (int64_t(1) << 31);
}

// The persistent GEMMs number their 128 x 256 output tiles with 32-bit ints:
// logits [N, V], dW [V, H] and dX [N, H] must each have fewer than 2^31 tiles.
inline bool tiles_ok(int64_t N, int64_t H, int64_t V) {
  const auto tiles = [](int64_t m, int64_t n) { return ((m + 127) / 128) * ((n + 255) / 256); };
  const int64_t lim = int64_t(1) << 31;
  return tiles(N, V) < lim && tiles(V, H) < lim && tiles(N, H) < lim;
}

// X, W and targets of an LM-head call: shapes, dtype, alignment.
inline vp_status check_inputs(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H,
                              int64_t V, int T, vp_dtype dtype) {
  if (!X || !W || !targets || !dtype_ok(dtype) || !shape_ok(N, H, V, T)) return VP_ERR_INVALID_ARG;
  if (!tiles_ok(N, H, V)) return VP_ERR_UNSUPPORTED;
  if (!aligned16(X) || !aligned16(W) || (H * esize_of(dtype)) % 16 != 0) return VP_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(targets) & 7u) != 0) return VP_ERR_UNSUPPORTED;
  return VP_OK;
}

// The same plus a caller workspace (non-NULL, 16-byte aligned).
inline vp_status check_args(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                            int T, vp_dtype dtype, const void* ws) {
  const vp_status st = check_inputs(X, W, targets, N, H, V, T, dtype);
  if (st != VP_OK) return st;
  if (!ws) return VP_ERR_INVALID_ARG;
  if (!aligned16(ws)) return VP_ERR_UNSUPPORTED;
  return VP_OK;
}

// Forward scratch: status header | (m, R) records [ntiles * maxseg][N] | z_y [N].
struct FwdLayout {
  int tile_v, maxseg;
  int64_t ntiles;
  size_t off_partial, off_zy, total;
};
inline FwdLayout fwd_layout(int64_t N, int64_t V, int T, vp_dtype dt) {
  FwdLayout L;
  const int64_t Vs = V / T;
  L.tile_v = dt == VP_BF16 ? kBf16TileV : kF32TileV;
  L.maxseg = dt == VP_BF16 ? lse_maxseg(V, Vs, T) : f32_maxseg(V, Vs, T);
  L.ntiles = (V + L.tile_v - 1) / L.tile_v;
  L.off_partial = kHeader;
  L.off_zy = align_up(L.off_partial + size_t(L.ntiles) * L.maxseg * N * sizeof(float2), kAlign);
  L.total = align_up(L.off_zy + size_t(N) * sizeof(float), kAlign);
  return L;
}

}  // namespace vp
