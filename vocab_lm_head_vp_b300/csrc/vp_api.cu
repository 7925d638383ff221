// libvp C ABI: argument validation, workspace layout and kernel dispatch for
// the vocab-parallel embedding and the fused LM head + cross-entropy.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/vp.h"
#include "../../include/vp_testing.h"
#include "vp_internal.h"

#define VP_EXPORT extern "C" __attribute__((visibility("default")))

namespace vp {

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

namespace {

// ---------------- backward workspace: header | g | dZ chunk | dX fp32 partial (bf16, >1 chunk)
struct BwdLayout {
  int64_t Vc, ldz, ldxt;
  size_t off_g, off_dz, off_acc, off_sk, off_xt, total;
};
int bwd_tile(vp_dtype dt) { return dt == VP_BF16 ? kBf16TileV : kF32TileV; }
BwdLayout bwd_layout_for_chunk(int64_t N, int64_t H, int64_t V, vp_dtype dt, int64_t Vc) {
  BwdLayout L;
  L.Vc = Vc;
  L.ldz = (Vc + 7) / 8 * 8;
  L.off_g = kHeader;
  L.off_dz = align_up(L.off_g + size_t(N) * sizeof(float), kAlign);
  L.off_acc = align_up(L.off_dz + size_t(N) * L.ldz * esize_of(dt), kAlign);
  const bool need_acc = dt == VP_BF16 && Vc < V;
  L.off_sk = align_up(L.off_acc + (need_acc ? size_t(N) * H * sizeof(float) : 0), kAlign);
  L.off_xt = align_up(L.off_sk + (dt == VP_BF16 ? sk_workspace_bytes() : 0), kAlign);
  L.ldxt = (N + 7) / 8 * 8;   // X^T [H][ldxt] bf16, for the dW GEMMs
  L.total = align_up(L.off_xt + (dt == VP_BF16 ? size_t(H) * L.ldxt * 2 : 0), kAlign);
  return L;
}
// Largest chunk that fits in ws bytes (0 if none does): all V, else the most
// whole tiles (the layout grows with the chunk, so a binary search over the
// tile count is exact whatever the sections' alignment).
int64_t bwd_chunk_from_ws(int64_t N, int64_t H, int64_t V, vp_dtype dt, size_t ws) {
  if (bwd_layout_for_chunk(N, H, V, dt, V).total <= ws) return V;
  const int64_t tile = bwd_tile(dt);
  int64_t lo = 0, hi = (V - 1) / tile;   // tiles per chunk, below V
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (bwd_layout_for_chunk(N, H, V, dt, mid * tile).total <= ws)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo * tile;
}

// ---------------- fused workspace (bf16), token chunk Nc:
// header | g [N] | records [ntiles*maxseg][Nc] | z_y [Nc] | tmax [ntiles][Nc] | P, then dZ, [Nc][ldp] 2-byte
struct FusedLayout {
  int64_t Nc, ldp, ntiles, ldxt;
  int maxseg;
  size_t off_g, off_partial, off_zy, off_tmax, off_p, off_sk, off_xt, total;
};
FusedLayout fused_layout(int64_t N, int64_t H, int64_t V, int T, int64_t Nc) {
  FusedLayout L;
  L.Nc = Nc;
  L.ldp = (V + 7) / 8 * 8;
  L.ntiles = (V + kBf16TileV - 1) / kBf16TileV;
  L.maxseg = lse_maxseg(V, V / T, T);
  L.off_g = kHeader;
  L.off_partial = align_up(L.off_g + size_t(N) * sizeof(float), kAlign);
  L.off_zy = align_up(L.off_partial + size_t(L.ntiles) * L.maxseg * Nc * sizeof(float2), kAlign);
  L.off_tmax = align_up(L.off_zy + size_t(Nc) * sizeof(float), kAlign);
  L.off_p = align_up(L.off_tmax + size_t(L.ntiles) * Nc * sizeof(float), kAlign);
  L.off_sk = align_up(L.off_p + size_t(Nc) * L.ldp * 2, kAlign);
  L.off_xt = align_up(L.off_sk + sk_workspace_bytes(), kAlign);
  L.ldxt = (Nc + 7) / 8 * 8;   // X_c^T [H][ldxt] bf16, for the dW GEMMs
  L.total = align_up(L.off_xt + size_t(H) * L.ldxt * 2, kAlign);
  return L;
}
constexpr int64_t kFusedRowAlign = 128;   // token chunks are whole 128-row GEMM blocks

// Budget of the fused call's saved probabilities when the caller names no
// token chunk: N_c x round8(V) 2-byte values stay below it (the logits are
// never held for all N tokens at once).  1.25 GiB: at V = 128256 the chunk
// that balanced_token_chunk picks within it holds 4608 tokens (1.18 GB).
constexpr size_t kFusedDefaultSavedBytes = size_t(5) << 28;

int64_t fused_default_chunk(int64_t N, int64_t V) {
  const size_t per_row = size_t((V + 7) / 8 * 8) * 2;
  int64_t nc = int64_t(kFusedDefaultSavedBytes / per_row) / kFusedRowAlign * kFusedRowAlign;
  if (nc < kFusedRowAlign) nc = kFusedRowAlign;
  return nc >= N ? N : nc;
}

// Token chunk of the fused call for at most nc_max rows per chunk.  Each
// chunk's dX GEMM runs in whole waves of the persistent grid (dx_plan), so
// equal chunks can leave a mostly idle last wave in every chunk: among chunk
// sizes from nc_max down to half of it (128-row blocks), take the one with the
// lowest total dX cost plus a quarter wave per chunk after the first (its fp32
// read-modify-write of dW), fewer chunks on a tie.
int64_t balanced_token_chunk(int64_t N, int64_t H, int64_t nc_max) {
  if (nc_max >= N) return N;
  const int64_t mmax = nc_max / kFusedRowAlign;
  int64_t best = mmax, best_k = -1;
  double best_cost = 0.0;
  for (int64_t m = mmax; m >= 1 && 2 * m >= mmax; --m) {
    const int64_t nc = m * kFusedRowAlign, k = (N + nc - 1) / nc;
    const double cost = static_cast<double>(k - 1) * (dx_plan(nc, H).cost + 0.25) + dx_plan(N - (k - 1) * nc, H).cost;
    if (best_k < 0 || cost < best_cost - 1e-9 || (cost < best_cost + 1e-9 && k < best_k)) {
      best = m;
      best_k = k;
      best_cost = cost;
    }
  }
  return best * kFusedRowAlign;
}

// Vocab chunk of the split backward for at most vc_max ids per chunk: the
// fewest chunks, as equal as the tile allows.
int64_t balanced_vocab_chunk(int64_t V, int64_t vc_max, int64_t tile) {
  if (vc_max >= V) return V;
  const int64_t k = (V + vc_max - 1) / vc_max;
  const int64_t vc = ((V + k - 1) / k + tile - 1) / tile * tile;
  return vc < vc_max ? vc : vc_max;
}

// Default vocab chunk of the split backward: one shard, V/T ids, rounded up
// to the tile (the pages' unit: each rank forms dZ for its own shard).
int64_t bwd_default_chunk(int64_t V, int T, vp_dtype dt) {
  const int64_t tile = bwd_tile(dt);
  const int64_t vc = (V / T + tile - 1) / tile * tile;
  return vc >= V ? V : vc;
}
// Largest token chunk that fits in ws bytes: all N, else a multiple of 128 (0
// if none fits).  The layout grows with the chunk, so a binary search over the
// 128-row block count is exact; an estimate from the size of one row misjudges
// small workspaces, where the sections' 256-byte alignment weighs.
int64_t fused_chunk_from_ws(int64_t N, int64_t H, int64_t V, int T, size_t ws) {
  if (fused_layout(N, H, V, T, N).total <= ws) return N;
  int64_t lo = 0, hi = (N - 1) / kFusedRowAlign;   // 128-row blocks per chunk, below N
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (fused_layout(N, H, V, T, mid * kFusedRowAlign).total <= ws)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo * kFusedRowAlign;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

constexpr int kMergeKernels = 1;   // lse_merge: the per-shard and the per-token steps in one kernel

// ---------------- optional per-launch event timing (vp_stage_timing_enable)
enum Stage {
  kEmbed, kLseGemm, kMerge, kMean, kScale, kDzGemm, kDwGemm, kDxGemm, kLsePGemm, kDzFromP, kEmbedBwd, kXT,
  kEmbedSort, kNumStages
};
const char* const kStageNames[kNumStages] = {"embed_gather",   "lse_stats_gemm",    "lse_merge", "loss_mean",
                                             "upstream_scale", "dz_recompute_gemm", "dw_gemm",   "dx_gemm",
                                             "lse_p_gemm",     "dz_from_p",         "embed_bwd", "x_transpose",
                                             "embed_bwd_sort"};
struct StageTimer {
  int cap = 0, used = 0;
  int dropped = 0;            // timed regions past `cap`, not recorded
  cudaEvent_t* ev = nullptr;  // 2 per launch
  int* stage = nullptr;
  int* kernels = nullptr;   // kernels launched inside each timed region
} g_timer;

// kernels_after: where the launch leaves the number of kernels it launched
// (read after it returns), for launches whose count depends on the shapes.
template <class F>
cudaError_t timed(Stage st, cudaStream_t s, F&& launch, int kernels = 1, const int* kernels_after = nullptr) {
  int slot = -1;
  if (g_timer.cap > 0 && g_timer.used >= g_timer.cap) ++g_timer.dropped;
  if (g_timer.cap > 0 && g_timer.used < g_timer.cap) {
    slot = g_timer.used++;
    g_timer.stage[slot] = st;
    g_timer.kernels[slot] = kernels;
    cudaEventRecord(g_timer.ev[2 * slot], s);
  }
  cudaError_t e = launch();
  if (slot >= 0) {
    if (kernels_after) g_timer.kernels[slot] = *kernels_after;
    cudaEventRecord(g_timer.ev[2 * slot + 1], s);
  }
  return e;
}

// dW_c (+)= dZ_c^T X: through X^T (transposed once into `xt` by the caller)
// when the GEMM form allows, else directly.
cudaError_t dw_gemm(const void* dz, int64_t ldz, const void* X, const void* xt, int64_t ldxt, int64_t N, int64_t H,
                    int64_t c0, int64_t Vc, float* dW, bool accumulate, uint32_t* status, cudaStream_t s) {
  if (dw_through_xt()) return bf16_dwt_chunk(xt, ldxt, dz, ldz, N, H, c0, Vc, dW, accumulate, status, s);
  return bf16_dw_chunk(dz, ldz, X, N, H, c0, Vc, dW, accumulate, status, s);
}

}  // namespace
}  // namespace vp

using namespace vp;

VP_EXPORT const char* vp_status_string(vp_status s) {
  switch (s) {
    case VP_OK: return "VP_OK";
    case VP_ERR_INVALID_ARG: return "VP_ERR_INVALID_ARG";
    case VP_ERR_UNSUPPORTED: return "VP_ERR_UNSUPPORTED";
    case VP_ERR_WORKSPACE: return "VP_ERR_WORKSPACE";
    case VP_ERR_CUDA: return "VP_ERR_CUDA";
  }
  return "VP_ERR_UNKNOWN";
}

VP_EXPORT const char* vp_version(void) { return "libvp 0.1 sm_103a"; }

VP_EXPORT vp_status vp_embed_fwd(const int64_t* ids, const void* W, void* out, int64_t N, int64_t H, int64_t V, int T,
                                 vp_dtype dtype, void* stream) {
  if (!ids || !W || !out || !dtype_ok(dtype) || !shape_ok(N, H, V, T)) return VP_ERR_INVALID_ARG;
  const int es = esize_of(dtype);
  if (!aligned16(W) || !aligned16(out) || (H * es) % 16 != 0) return VP_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(ids) & 7u) != 0) return VP_ERR_UNSUPPORTED;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = timed(kEmbed, s, [&] { return embed_gather(ids, W, out, N, H, V, V / T, T, es, s); });
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_embed_fwd_sp(const int64_t* ids, const void* W, void* out, int64_t N, int64_t H, int64_t V,
                                    int T, int rank, vp_dtype dtype, void* stream) {
  if (!ids || !W || !out || !dtype_ok(dtype) || !shape_ok(N, H, V, T)) return VP_ERR_INVALID_ARG;
  if (N % T != 0 || rank < 0 || rank >= T) return VP_ERR_INVALID_ARG;
  const int es = esize_of(dtype);
  if (!aligned16(W) || !aligned16(out) || (H * es) % 16 != 0) return VP_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(ids) & 7u) != 0) return VP_ERR_UNSUPPORTED;
  cudaStream_t s = as_stream(stream);
  const int64_t rows = N / T;
  // rank's token slice of the shard sum: the gather of exactly those tokens
  cudaError_t e =
      timed(kEmbed, s, [&] { return embed_gather(ids + rank * rows, W, out, rows, H, V, V / T, T, es, s); });
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT size_t vp_embed_bwd_workspace_size(int64_t N, int64_t H, int64_t V, int T, vp_dtype dtype) {
  if (!dtype_ok(dtype) || !shape_ok(N, H, V, T)) return 0;
  return align_up(embed_bwd_workspace(N, H), kAlign);
}

static vp_status check_embed_bwd(const void* dOut, const float* dW, int64_t N, int64_t H, int64_t V, int T,
                                 vp_dtype dtype, const void* workspace, size_t ws_bytes) {
  if (!dOut || !dW || !workspace || !dtype_ok(dtype) || !shape_ok(N, H, V, T)) return VP_ERR_INVALID_ARG;
  const int es = esize_of(dtype);
  if (!aligned16(dOut) || !aligned16(dW) || !aligned16(workspace) || (H * es) % 16 != 0) return VP_ERR_UNSUPPORTED;
  if (ws_bytes < embed_bwd_workspace(N, H)) return VP_ERR_WORKSPACE;
  return VP_OK;
}

VP_EXPORT vp_status vp_embed_bwd_plan(const int64_t* ids, int64_t N, int64_t H, int64_t V, int T, void* workspace,
                                      size_t ws_bytes, void* stream) {
  if (!ids || !workspace || !shape_ok(N, H, V, T)) return VP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ids) & 7u) != 0 || !aligned16(workspace)) return VP_ERR_UNSUPPORTED;
  if (ws_bytes < embed_bwd_workspace(N, H)) return VP_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = timed(kEmbedSort, s, [&] { return embed_bwd_sort(ids, N, V, workspace, s); },
                        embed_bwd_sort_kernels(N));
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_embed_bwd_planned(const void* dOut, float* dW, int64_t N, int64_t H, int64_t V, int T,
                                         vp_dtype dtype, int accumulate, void* workspace, size_t ws_bytes,
                                         void* stream) {
  const vp_status st = check_embed_bwd(dOut, dW, N, H, V, T, dtype, workspace, ws_bytes);
  if (st != VP_OK) return st;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = timed(kEmbedBwd, s, [&] {
    return embed_bwd_sums(dOut, dW, N, H, V, esize_of(dtype), accumulate != 0, workspace, s);
  }, 2);
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_embed_bwd(const int64_t* ids, const void* dOut, float* dW, int64_t N, int64_t H, int64_t V,
                                 int T, vp_dtype dtype, int accumulate, void* workspace, size_t ws_bytes,
                                 void* stream) {
  if (!ids) return VP_ERR_INVALID_ARG;
  vp_status st = check_embed_bwd(dOut, dW, N, H, V, T, dtype, workspace, ws_bytes);
  if (st != VP_OK) return st;
  if ((reinterpret_cast<uintptr_t>(ids) & 7u) != 0) return VP_ERR_UNSUPPORTED;
  st = vp_embed_bwd_plan(ids, N, H, V, T, workspace, ws_bytes, stream);
  if (st != VP_OK) return st;
  return vp_embed_bwd_planned(dOut, dW, N, H, V, T, dtype, accumulate, workspace, ws_bytes, stream);
}

VP_EXPORT size_t vp_lmhead_ce_workspace_size(int64_t N, int64_t H, int64_t V, int T, vp_dtype dtype, int pass,
                                             int64_t chunk) {
  if (!dtype_ok(dtype) || !shape_ok(N, H, V, T)) return 0;
  if (pass == 0) return fwd_layout(N, V, T, dtype).total;
  if (pass == 2 && dtype == VP_BF16) {
    int64_t nc = chunk <= 0 ? balanced_token_chunk(N, H, fused_default_chunk(N, V)) : chunk;
    if (nc < N) {
      nc = nc / kFusedRowAlign * kFusedRowAlign;
      if (nc < kFusedRowAlign) nc = kFusedRowAlign;
    }
    if (nc > N) nc = N;
    return fused_layout(N, H, V, T, nc).total;
  }
  if (pass == 3 && dtype == VP_BF16) return fused_layout(N, H, V, T, N).total;   // kept forward state, all N
  if (pass == 2 || pass == 3) {   // fp32: the forward, then the recompute backward in the same bytes
    const size_t f = fwd_layout(N, V, T, dtype).total;
    const size_t b = vp_lmhead_ce_workspace_size(N, H, V, T, dtype, 1, chunk);
    return f > b ? f : b;
  }
  if (pass != 1) return 0;
  int64_t vc = chunk <= 0 ? bwd_default_chunk(V, T, dtype) : chunk;
  if (vc < V) {
    const int64_t tile = bwd_tile(dtype);
    vc = (vc + tile - 1) / tile * tile;
  }
  if (vc > V) vc = V;
  return bwd_layout_for_chunk(N, H, V, dtype, vc).total;
}

static vp_status check_common(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                              int T, vp_dtype dtype, const void* ws) {
  vp_status st = check_args(X, W, targets, N, H, V, T, dtype, ws);
  if (st != VP_OK) return st;
  if (dtype == VP_BF16 && !tensor_map_encoder()) return VP_ERR_CUDA;
  return VP_OK;
}

VP_EXPORT vp_status vp_lmhead_ce_fwd(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H,
                                     int64_t V, int T, int64_t ignore_index, vp_dtype dtype, float* loss, float* lse,
                                     float* loss_mean, float* shard_stats, int32_t* n_bad, void* workspace,
                                     size_t ws_bytes, void* stream) {
  if (!loss || !lse) return VP_ERR_INVALID_ARG;
  vp_status st = check_common(X, W, targets, N, H, V, T, dtype, workspace);
  if (st != VP_OK) return st;
  const FwdLayout L = fwd_layout(N, V, T, dtype);
  if (ws_bytes < L.total) return VP_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float2* partial = reinterpret_cast<float2*>(ws + L.off_partial);
  float* zy = reinterpret_cast<float*>(ws + L.off_zy);
  const int64_t Vs = V / T;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) {
    e = timed(kLseGemm, s, [&] {
      if (dtype == VP_BF16) return bf16_lse_stats(X, W, targets, N, H, V, Vs, partial, L.maxseg, zy, status, s);
      return f32_lse_stats(static_cast<const float*>(X), static_cast<const float*>(W), targets, N, H, V, Vs,
                           partial, L.maxseg, zy, s);
    });
  }
  if (e == cudaSuccess)
    e = timed(kMerge, s, [&] {
      return lse_merge(partial, zy, targets, N, V, Vs, T, L.tile_v, L.maxseg, ignore_index, loss, lse, shard_stats,
                       status, s);
    }, kMergeKernels);
  if (e == cudaSuccess && (loss_mean || n_bad))
    e = timed(kMean, s, [&] { return loss_mean_and_bad(loss, targets, N, V, ignore_index, loss_mean, n_bad, s); });
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_lmhead_ce_bwd(const void* X, const void* W, const int64_t* targets, const float* lse,
                                     const float* dloss, const float* dmean, int64_t N, int64_t H, int64_t V,
                                     int T,
                                     int64_t ignore_index, vp_dtype dtype, void* dX, float* dW, void* workspace,
                                     size_t ws_bytes, void* stream) {
  if (!lse || !dX || !dW) return VP_ERR_INVALID_ARG;
  vp_status st = check_common(X, W, targets, N, H, V, T, dtype, workspace);
  if (st != VP_OK) return st;
  if (!aligned16(dX) || !aligned16(dW)) return VP_ERR_UNSUPPORTED;
  const int64_t Vc_max = bwd_chunk_from_ws(N, H, V, dtype, ws_bytes);
  if (Vc_max <= 0) return VP_ERR_WORKSPACE;
  const int64_t Vc = balanced_vocab_chunk(V, Vc_max, bwd_tile(dtype));
  const BwdLayout L = bwd_layout_for_chunk(N, H, V, dtype, Vc);
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* g = reinterpret_cast<float*>(ws + L.off_g);
  void* dz = ws + L.off_dz;
  float* acc = reinterpret_cast<float*>(ws + L.off_acc);
  float* skw = reinterpret_cast<float*>(ws + L.off_sk);
  void* xt = ws + L.off_xt;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = timed(kScale, s, [&] { return upstream_scale(targets, dloss, dmean, N, V, ignore_index, g, s); });
  if (e == cudaSuccess && dtype == VP_BF16 && dw_through_xt())
    e = timed(kXT, s, [&] { return transpose_bf16(X, N, H, H, xt, L.ldxt, s); });
  const bool single = Vc >= V;
  for (int64_t c0 = 0; c0 < V && e == cudaSuccess; c0 += Vc) {
    const int64_t vc = (V - c0) < Vc ? (V - c0) : Vc;
    const bool first = c0 == 0, last = c0 + vc >= V;
    if (dtype == VP_BF16) {
      e = timed(kDzGemm, s, [&] { return bf16_dz_chunk(X, W, targets, lse, g, N, H, c0, vc, dz, L.ldz, status, s); });
      if (e == cudaSuccess)
        e = timed(kDwGemm, s,
                  [&] { return dw_gemm(dz, L.ldz, X, xt, L.ldxt, N, H, c0, vc, dW, false, status, s); });
      if (e == cudaSuccess) {
        // dX over chunks: bf16 store (one chunk), else fp32 store / fp32 add / bf16 = fp32 partial + last
        void* out = (single || last) ? dX : static_cast<void*>(acc);
        const int mode = single ? 3 : first ? 0 : !last ? 1 : 2;
        int nk = 1;
        e = timed(kDxGemm, s, [&] {
          return bf16_dx_chunk(dz, L.ldz, W, N, H, c0, vc, out, mode == 2 ? acc : nullptr, mode, status, s, skw, &nk);
        }, 1, &nk);
      }
    } else {
      const float* Xf = static_cast<const float*>(X);
      const float* Wf = static_cast<const float*>(W);
      float* dzf = static_cast<float*>(dz);
      e = timed(kDzGemm, s, [&] { return f32_dz_chunk(Xf, Wf, targets, lse, g, N, H, c0, vc, dzf, L.ldz, s); });
      // dW[c0+v, h] = sum_n dZ[n, v] X[n, h]
      if (e == cudaSuccess)
        e = timed(kDwGemm, s, [&] { return f32_gemm(dzf, 1, L.ldz, Xf, H, 1, dW + c0 * H, H, vc, H, N, false, s); });
      // dX[n, h] (+)= sum_v dZ[n, v] W[c0+v, h]
      if (e == cudaSuccess)
        e = timed(kDxGemm, s, [&] {
          return f32_gemm(dzf, L.ldz, 1, Wf + c0 * H, H, 1, static_cast<float*>(dX), H, N, H, vc, !first, s);
        });
    }
  }
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_lmhead_ce_fwd_bwd(const void* X, const void* W, const int64_t* targets, const float* dloss,
                                         const float* dmean, int64_t N, int64_t H, int64_t V, int T, int64_t ignore_index,
                                         vp_dtype dtype, float* loss, float* lse, float* loss_mean,
                                         float* shard_stats, int32_t* n_bad, void* dX, float* dW, void* workspace,
                                         size_t ws_bytes, void* stream) {
  if (!loss || !lse || !dX || !dW) return VP_ERR_INVALID_ARG;
  vp_status st = check_args(X, W, targets, N, H, V, T, dtype, workspace);
  if (st != VP_OK) return st;
  if (!aligned16(dX) || !aligned16(dW)) return VP_ERR_UNSUPPORTED;
  if (dtype == VP_F32) {
    // CUDA-core fp32 path: the forward, then the recompute backward, both in this workspace
    if (ws_bytes < fwd_layout(N, V, T, dtype).total || bwd_chunk_from_ws(N, H, V, dtype, ws_bytes) <= 0)
      return VP_ERR_WORKSPACE;
    st = vp_lmhead_ce_fwd(X, W, targets, N, H, V, T, ignore_index, dtype, loss, lse, loss_mean, shard_stats, n_bad,
                          workspace, ws_bytes, stream);
    if (st != VP_OK) return st;
    return vp_lmhead_ce_bwd(X, W, targets, lse, dloss, dmean, N, H, V, T, ignore_index, dtype, dX, dW, workspace,
                            ws_bytes, stream);
  }
  const int64_t Nc_max = fused_chunk_from_ws(N, H, V, T, ws_bytes);
  if (Nc_max <= 0) return VP_ERR_WORKSPACE;
  const int64_t Nc = balanced_token_chunk(N, H, Nc_max);
  if (!tensor_map_encoder()) return VP_ERR_CUDA;
  const FusedLayout L = fused_layout(N, H, V, T, Nc);
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* g = reinterpret_cast<float*>(ws + L.off_g);
  float2* partial = reinterpret_cast<float2*>(ws + L.off_partial);
  float* zy = reinterpret_cast<float*>(ws + L.off_zy);
  float* tmax = reinterpret_cast<float*>(ws + L.off_tmax);
  void* P = ws + L.off_p;
  float* skw = reinterpret_cast<float*>(ws + L.off_sk);
  void* xt = ws + L.off_xt;
  const int64_t Vs = V / T;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = timed(kScale, s, [&] { return upstream_scale(targets, dloss, dmean, N, V, ignore_index, g, s); });
  for (int64_t n0 = 0; n0 < N && e == cudaSuccess; n0 += Nc) {
    const int64_t nc = (N - n0) < Nc ? (N - n0) : Nc;
    const void* Xc = static_cast<const uint8_t*>(X) + n0 * H * 2;
    const int64_t* yc = targets + n0;
    e = timed(kLsePGemm, s, [&] {
      return bf16_lse_stats_p(Xc, W, yc, nc, H, V, Vs, partial, L.maxseg, zy, tmax, P, L.ldp, status, s);
    });
    if (e == cudaSuccess)
      e = timed(kMerge, s, [&] {
        return lse_merge_ld(partial, zy, yc, nc, V, Vs, T, kBf16TileV, L.maxseg, ignore_index, loss + n0, lse + n0,
                            shard_stats ? shard_stats + n0 : nullptr, N, status, s);
      }, kMergeKernels);
    void* dXc = static_cast<uint8_t*>(dX) + n0 * H * 2;
    // p -> dZ in place, then dW = sum over token chunks of dZ_c^T X_c; dX rows of this chunk are complete
    if (e == cudaSuccess)
      e = timed(kDzFromP, s, [&] { return dz_from_p(P, L.ldp, tmax, lse + n0, g + n0, yc, nc, V, s); });
    if (e == cudaSuccess)
      e = timed(kXT, s, [&] { return dw_through_xt() ? transpose_bf16(Xc, nc, H, H, xt, L.ldxt, s) : cudaSuccess; },
                dw_through_xt() ? 1 : 0);
    if (e == cudaSuccess)
      e = timed(kDwGemm, s,
                [&] { return dw_gemm(P, L.ldp, Xc, xt, L.ldxt, nc, H, 0, V, dW, n0 > 0, status, s); });
    int nk = 1;
    if (e == cudaSuccess)
      e = timed(kDxGemm, s, [&] {
        return bf16_dx_chunk(P, L.ldp, W, nc, H, 0, V, dXc, nullptr, 3, status, s, skw, &nk);
      }, 1, &nk);
  }
  if (e == cudaSuccess && (loss_mean || n_bad))
    e = timed(kMean, s, [&] { return loss_mean_and_bad(loss, targets, N, V, ignore_index, loss_mean, n_bad, s); });
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_lmhead_ce_fwd_keep(const void* X, const void* W, const int64_t* targets, int64_t N,
                                          int64_t H, int64_t V, int T, int64_t ignore_index, vp_dtype dtype,
                                          float* loss, float* lse, float* loss_mean, float* shard_stats,
                                          int32_t* n_bad, void* saved, size_t saved_bytes, void* stream) {
  if (!loss || !lse) return VP_ERR_INVALID_ARG;
  vp_status st = check_args(X, W, targets, N, H, V, T, dtype, saved);
  if (st != VP_OK) return st;
  if (dtype == VP_F32)   // fp32: nothing is kept; the backward recomputes in the same bytes
    return vp_lmhead_ce_fwd(X, W, targets, N, H, V, T, ignore_index, dtype, loss, lse, loss_mean, shard_stats, n_bad,
                            saved, saved_bytes, stream);
  const FusedLayout L = fused_layout(N, H, V, T, N);
  if (saved_bytes < L.total) return VP_ERR_WORKSPACE;
  if (!tensor_map_encoder()) return VP_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(saved);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float2* partial = reinterpret_cast<float2*>(ws + L.off_partial);
  float* zy = reinterpret_cast<float*>(ws + L.off_zy);
  float* tmax = reinterpret_cast<float*>(ws + L.off_tmax);
  void* P = ws + L.off_p;
  const int64_t Vs = V / T;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = timed(kLsePGemm, s, [&] {
      return bf16_lse_stats_p(X, W, targets, N, H, V, Vs, partial, L.maxseg, zy, tmax, P, L.ldp, status, s);
    });
  if (e == cudaSuccess)
    e = timed(kMerge, s, [&] {
      return lse_merge(partial, zy, targets, N, V, Vs, T, kBf16TileV, L.maxseg, ignore_index, loss, lse, shard_stats,
                       status, s);
    }, kMergeKernels);
  if (e == cudaSuccess && (loss_mean || n_bad))
    e = timed(kMean, s, [&] { return loss_mean_and_bad(loss, targets, N, V, ignore_index, loss_mean, n_bad, s); });
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_lmhead_ce_bwd_saved(const void* X, const void* W, const int64_t* targets, const float* lse,
                                           const float* dloss, const float* dmean, int64_t N, int64_t H, int64_t V,
                                           int T, int64_t ignore_index, vp_dtype dtype, void* dX, float* dW,
                                           void* saved, size_t saved_bytes, void* stream) {
  if (!lse || !dX || !dW) return VP_ERR_INVALID_ARG;
  vp_status st = check_args(X, W, targets, N, H, V, T, dtype, saved);
  if (st != VP_OK) return st;
  if (!aligned16(dX) || !aligned16(dW)) return VP_ERR_UNSUPPORTED;
  if (dtype == VP_F32)
    return vp_lmhead_ce_bwd(X, W, targets, lse, dloss, dmean, N, H, V, T, ignore_index, dtype, dX, dW, saved,
                            saved_bytes, stream);
  const FusedLayout L = fused_layout(N, H, V, T, N);
  if (saved_bytes < L.total) return VP_ERR_WORKSPACE;
  if (!tensor_map_encoder()) return VP_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(saved);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* g = reinterpret_cast<float*>(ws + L.off_g);
  float* tmax = reinterpret_cast<float*>(ws + L.off_tmax);
  void* P = ws + L.off_p;
  float* skw = reinterpret_cast<float*>(ws + L.off_sk);
  void* xt = ws + L.off_xt;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = timed(kScale, s, [&] { return upstream_scale(targets, dloss, dmean, N, V, ignore_index, g, s); });
  // p becomes dZ in place, scaled per row and tile by c = g exp(tmax - lse) from the kept tile maxima
  if (e == cudaSuccess) e = timed(kDzFromP, s, [&] { return dz_from_p(P, L.ldp, tmax, lse, g, targets, N, V, s); });
  if (e == cudaSuccess && dw_through_xt())
    e = timed(kXT, s, [&] { return transpose_bf16(X, N, H, H, xt, L.ldxt, s); });
  if (e == cudaSuccess)
    e = timed(kDwGemm, s, [&] { return dw_gemm(P, L.ldp, X, xt, L.ldxt, N, H, 0, V, dW, false, status, s); });
  int nk = 1;
  if (e == cudaSuccess)
    e = timed(kDxGemm, s, [&] { return bf16_dx_chunk(P, L.ldp, W, N, H, 0, V, dX, nullptr, 3, status, s, skw, &nk); },
              1, &nk);
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

// ---------------- one shard of a T-rank vocabulary (a rank that holds only W_t)
static vp_status check_shard(const void* X, const void* W_t, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                             int T, int t, vp_dtype dtype, const void* ws) {
  if (!shape_ok(N, H, V, T) || t < 0 || t >= T) return VP_ERR_INVALID_ARG;
  return check_args(X, W_t, targets, N, H, V / T, 1, dtype, ws);
}

VP_EXPORT vp_status vp_lmhead_ce_shard_fwd(const void* X, const void* W_t, const int64_t* targets, int64_t N,
                                           int64_t H, int64_t V, int T, int t, int64_t ignore_index, vp_dtype dtype,
                                           float* stats, void* workspace, size_t ws_bytes, void* stream) {
  if (!stats) return VP_ERR_INVALID_ARG;
  vp_status st = check_shard(X, W_t, targets, N, H, V, T, t, dtype, workspace);
  if (st != VP_OK) return st;
  if (dtype == VP_BF16 && !tensor_map_encoder()) return VP_ERR_CUDA;
  const int64_t Vs = V / T;
  const FwdLayout L = fwd_layout(N, Vs, 1, dtype);   // the shard alone: one record per tile
  if (ws_bytes < L.total) return VP_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float2* partial = reinterpret_cast<float2*>(ws + L.off_partial);
  float* zy = reinterpret_cast<float*>(ws + L.off_zy);
  const int64_t start = static_cast<int64_t>(t) * Vs;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = timed(kLseGemm, s, [&] {
      if (dtype == VP_BF16)
        return bf16_lse_stats(X, W_t, targets, N, H, Vs, Vs, partial, L.maxseg, zy, status, s, start);
      return f32_lse_stats(static_cast<const float*>(X), static_cast<const float*>(W_t), targets, N, H, Vs, Vs,
                           partial, L.maxseg, zy, s, start);
    });
  if (e == cudaSuccess)
    e = timed(kMerge, s, [&] {
      return shard_stats(partial, zy, targets, N, V, start, Vs, L.ntiles, ignore_index, stats, status, s);
    });
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_lmhead_ce_merge_stats(const float* stats, const int64_t* targets, int64_t N, int64_t V, int T,
                                             int64_t ignore_index, float* loss, float* lse, float* loss_mean,
                                             int32_t* n_bad, void* stream) {
  if (!stats || !targets || !loss || !lse || N <= 0 || V <= 0 || T <= 0 || V % T != 0 || N >= (int64_t(1) << 31))
    return VP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(targets) & 7u) != 0) return VP_ERR_UNSUPPORTED;
  cudaStream_t s = as_stream(stream);
  cudaError_t e =
      timed(kMerge, s, [&] { return merge_shard_stats(stats, targets, N, V, T, ignore_index, loss, lse, s); });
  if (e == cudaSuccess && (loss_mean || n_bad))
    e = timed(kMean, s, [&] { return loss_mean_and_bad(loss, targets, N, V, ignore_index, loss_mean, n_bad, s); });
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_lmhead_ce_shard_bwd(const void* X, const void* W_t, const int64_t* targets, const float* lse,
                                           const float* dloss, const float* dmean, int64_t N, int64_t H, int64_t V,
                                           int T, int t, int64_t ignore_index, vp_dtype dtype, float* dX_t,
                                           float* dW_t, void* workspace, size_t ws_bytes, void* stream) {
  if (!lse || !dX_t || !dW_t) return VP_ERR_INVALID_ARG;
  vp_status st = check_shard(X, W_t, targets, N, H, V, T, t, dtype, workspace);
  if (st != VP_OK) return st;
  if (!aligned16(dX_t) || !aligned16(dW_t)) return VP_ERR_UNSUPPORTED;
  if (dtype == VP_BF16 && !tensor_map_encoder()) return VP_ERR_CUDA;
  const int64_t Vs = V / T;
  const int64_t Vc_max = bwd_chunk_from_ws(N, H, Vs, dtype, ws_bytes);
  if (Vc_max <= 0) return VP_ERR_WORKSPACE;
  const int64_t Vc = balanced_vocab_chunk(Vs, Vc_max, bwd_tile(dtype));
  const BwdLayout L = bwd_layout_for_chunk(N, H, Vs, dtype, Vc);
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* g = reinterpret_cast<float*>(ws + L.off_g);
  void* dz = ws + L.off_dz;
  float* skw = reinterpret_cast<float*>(ws + L.off_sk);
  void* xt = ws + L.off_xt;
  const int64_t start = static_cast<int64_t>(t) * Vs;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)   // validity against the whole vocabulary: every rank sees the same N_valid
    e = timed(kScale, s, [&] { return upstream_scale(targets, dloss, dmean, N, V, ignore_index, g, s); });
  if (e == cudaSuccess && dtype == VP_BF16 && dw_through_xt())
    e = timed(kXT, s, [&] { return transpose_bf16(X, N, H, H, xt, L.ldxt, s); });
  for (int64_t c0 = 0; c0 < Vs && e == cudaSuccess; c0 += Vc) {
    const int64_t vc = (Vs - c0) < Vc ? (Vs - c0) : Vc;
    const bool first = c0 == 0;
    if (dtype == VP_BF16) {
      e = timed(kDzGemm, s,
                [&] { return bf16_dz_chunk(X, W_t, targets, lse, g, N, H, c0, vc, dz, L.ldz, status, s, start); });
      if (e == cudaSuccess)
        e = timed(kDwGemm, s,
                  [&] { return dw_gemm(dz, L.ldz, X, xt, L.ldxt, N, H, c0, vc, dW_t, false, status, s); });
      // this shard's part of dX in fp32: stored by the first chunk, added by the others
      if (e == cudaSuccess) {
        int nk = 1;
        e = timed(kDxGemm, s, [&] {
          return bf16_dx_chunk(dz, L.ldz, W_t, N, H, c0, vc, dX_t, nullptr, first ? 0 : 1, status, s, skw, &nk);
        }, 1, &nk);
      }
    } else {
      const float* Xf = static_cast<const float*>(X);
      const float* Wf = static_cast<const float*>(W_t);
      float* dzf = static_cast<float*>(dz);
      e = timed(kDzGemm, s,
                [&] { return f32_dz_chunk(Xf, Wf, targets, lse, g, N, H, c0, vc, dzf, L.ldz, s, start); });
      if (e == cudaSuccess)
        e = timed(kDwGemm, s, [&] { return f32_gemm(dzf, 1, L.ldz, Xf, H, 1, dW_t + c0 * H, H, vc, H, N, false, s); });
      if (e == cudaSuccess)
        e = timed(kDxGemm, s, [&] { return f32_gemm(dzf, L.ldz, 1, Wf + c0 * H, H, 1, dX_t, H, N, H, vc, !first, s); });
    }
  }
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_read_device_status(const void* workspace, uint32_t* flags, void* stream) {
  if (!workspace || !flags) return VP_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e == cudaSuccess) e = cudaMemcpy(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_test_gemm_bf16(const void* A, const void* B, float* D, int64_t M, int64_t N, int64_t K,
                                      int a_mn_major, int b_mn_major, void* workspace, void* stream) {
  if (!A || !B || !D || !workspace || M <= 0 || N <= 0 || K <= 0) return VP_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !aligned16(workspace)) return VP_ERR_UNSUPPORTED;
  if ((a_mn_major ? M : K) % 8 != 0 || (b_mn_major ? N : K) % 8 != 0 || N % 4 != 0) return VP_ERR_UNSUPPORTED;
  if (!tensor_map_encoder()) return VP_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  uint32_t* status = static_cast<uint32_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = bf16_gemm_test(A, B, D, M, N, K, a_mn_major, b_mn_major, status, s);
  return e == cudaSuccess ? VP_OK : VP_ERR_CUDA;
}

VP_EXPORT vp_status vp_stage_timing_enable(int max_launches) {
  StageTimer& t = g_timer;
  if (t.ev) {
    for (int i = 0; i < 2 * t.cap; ++i) cudaEventDestroy(t.ev[i]);
    delete[] t.ev;
    delete[] t.stage;
    delete[] t.kernels;
    t.ev = nullptr;
    t.stage = nullptr;
    t.kernels = nullptr;
  }
  t.cap = 0;
  t.used = 0;
  t.dropped = 0;
  if (max_launches <= 0) return VP_OK;
  t.ev = new cudaEvent_t[2 * max_launches];
  t.stage = new int[max_launches];
  t.kernels = new int[max_launches];
  for (int i = 0; i < 2 * max_launches; ++i) {
    if (cudaEventCreate(&t.ev[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(t.ev[j]);
      delete[] t.ev;
      delete[] t.stage;
      delete[] t.kernels;
      t.ev = nullptr;
      t.stage = nullptr;
      t.kernels = nullptr;
      return VP_ERR_CUDA;
    }
  }
  t.cap = max_launches;
  return VP_OK;
}

VP_EXPORT int vp_stage_timing_read(float* ms, int32_t* counts, int n) {
  for (int s = 0; s < n && s < kNumStages; ++s) {
    if (ms) ms[s] = 0.f;
    if (counts) counts[s] = 0;
  }
  const StageTimer& t = g_timer;
  for (int i = 0; i < t.used; ++i) {
    float x = 0.f;
    if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess) return -1;
    if (cudaEventElapsedTime(&x, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess) return -1;
    const int s = t.stage[i];
    if (s < n) {
      if (ms) ms[s] += x;
      if (counts) counts[s] += t.kernels[i];
    }
  }
  return kNumStages;
}

VP_EXPORT int vp_stage_timing_dropped(void) { return g_timer.dropped; }

VP_EXPORT const char* vp_stage_name(int stage) {
  return (stage >= 0 && stage < kNumStages) ? kStageNames[stage] : nullptr;
}

VP_EXPORT vp_status vp_test_set_gemm_variant(int variant) {
  if (variant < 0 || variant > 3) return VP_ERR_INVALID_ARG;
  set_gemm_variant(variant);
  return VP_OK;
}

VP_EXPORT vp_status vp_test_dx_plan(int64_t rows, int64_t H, int sms, int32_t* tile_rows, int32_t* streamk,
                                    double* cost) {
  if (rows <= 0 || H <= 0 || sms <= 0 || !tile_rows || !streamk || !cost) return VP_ERR_INVALID_ARG;
  const DxPlan p = dx_plan_on(rows, H, sms);
  *tile_rows = p.rows;
  *streamk = p.streamk ? 1 : 0;
  *cost = p.cost;
  return VP_OK;
}

VP_EXPORT vp_status vp_test_set_wait_fault(int mode, uint64_t wait_ns) {
  if (mode < 0 || mode > 2) return VP_ERR_INVALID_ARG;
  set_wait_fault(mode, wait_ns);
  return VP_OK;
}
