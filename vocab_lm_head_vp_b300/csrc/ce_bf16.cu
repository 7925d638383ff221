// bf16 tensor-core path of the fused LM head + vocab-parallel cross-entropy:
// the three epilogues that ride on the tcgen05 GEMM core and their launchers.
//
//   EpiLseStats  forward: per token row and per shard segment of a 256-wide
//                vocab tile, the local max m and sum exp(z - m), plus the
//                target logit when the tile owns the target ("Vocab
//                Parallelism" sec. 5.3.1; interview note figure 2).
//   EpiDZ        backward: recomputed logits -> dZ = g (exp(z - lse) - 1[j=y])
//                stored as bf16 for one vocab chunk (sec. 5.3.2).
//   EpiStore     dX / dW: fp32 accumulator -> fp32 store, fp32 read-add-store,
//                or bf16 store (optionally adding an fp32 partial first).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "umma_gemm.cuh"
#include "vp_internal.h"

namespace vp {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ forward
struct EpiLseStats {
  struct Params {
    float2* partial;          // [num_vtiles * maxseg][N] (m, S)
    float* zy;                // [N] target logit, written by the owning tile
    const int64_t* targets;   // [N]
    int64_t N, V, Vs;         // tokens, vocab, shard width V/T
    int maxseg;               // record slots per vocab tile
  };
  __device__ static void run(const Params& p, uint32_t taddr, int64_t n, int /*mb*/, int nb) {
    const int64_t v0 = static_cast<int64_t>(nb) * kBN;
    const int64_t vend = min(v0 + kBN, p.V);
    const bool row_ok = n < p.N;
    const int64_t y = row_ok ? p.targets[n] : -1;
    const int64_t yl = y - v0;
    int64_t t = v0 / p.Vs;
    int64_t seg_end = min((t + 1) * p.Vs, vend);
    int k = 0;
    float m = -INFINITY, s = 0.f, zyv = 0.f;
    bool have_zy = false;
    float2* rec = p.partial + (static_cast<int64_t>(nb) * p.maxseg) * p.N + n;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int64_t c0 = v0 + c * 32;
      if (c0 >= vend) break;  // uniform over the CTA
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait();
      const int64_t j = yl - c * 32;
      if (j >= 0 && j < 32 && c0 + j < vend) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < 32; ++q) v = (q == j) ? as_f(r[q]) : v;
        zyv = v;
        have_zy = true;
      }
      if (c0 + 32 <= seg_end) {
        // whole chunk inside the current shard segment
        float cm = as_f(r[0]);
#pragma unroll
        for (int q = 1; q < 32; ++q) cm = fmaxf(cm, as_f(r[q]));
        if (cm > m) {
          s *= ex2_approx((m - cm) * kLog2e);
          m = cm;
        }
        const float mL = m * kLog2e;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          a0 += ex2_approx(fmaf(as_f(r[q + 0]), kLog2e, -mL));
          a1 += ex2_approx(fmaf(as_f(r[q + 1]), kLog2e, -mL));
          a2 += ex2_approx(fmaf(as_f(r[q + 2]), kLog2e, -mL));
          a3 += ex2_approx(fmaf(as_f(r[q + 3]), kLog2e, -mL));
        }
        s += (a0 + a1) + (a2 + a3);
      } else {
        // a shard edge or the vocab end falls inside this chunk
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int64_t col = c0 + q;
          if (col >= vend) break;
          if (col == seg_end) {
            if (row_ok) rec[static_cast<int64_t>(k) * p.N] = make_float2(m, s);
            ++k;
            ++t;
            seg_end = min((t + 1) * p.Vs, vend);
            m = -INFINITY;
            s = 0.f;
          }
          const float z = as_f(r[q]);
          if (z > m) {
            s = s * ex2_approx((m - z) * kLog2e) + 1.f;
            m = z;
          } else {
            s += ex2_approx((z - m) * kLog2e);
          }
        }
      }
    }
    if (row_ok) {
      rec[static_cast<int64_t>(k) * p.N] = make_float2(m, s);
      if (have_zy) p.zy[n] = zyv;
    }
  }
};

// ------------------------------------------------------------------ backward dZ
struct EpiDZ {
  struct Params {
    __nv_bfloat16* dz;        // [N][ldz], chunk-local columns
    int64_t ldz;
    const float* lse;         // [N]
    const float* g;           // [N] upstream scale (0 for ignored rows)
    const int64_t* targets;   // [N]
    int64_t N;
    int64_t c0, Vc;           // chunk start (global vocab id) and width
  };
  __device__ static void run(const Params& p, uint32_t taddr, int64_t n, int /*mb*/, int nb) {
    const int64_t v0 = static_cast<int64_t>(nb) * kBN;   // chunk-local
    const int64_t vend = min(v0 + kBN, p.Vc);
    const bool row_ok = n < p.N;
    const float g = row_ok ? p.g[n] : 0.f;
    const float nl = row_ok ? -p.lse[n] * kLog2e : 0.f;
    const int64_t yl = (row_ok ? p.targets[n] : -1) - p.c0 - v0;
    __nv_bfloat16* out = p.dz + (row_ok ? n : 0) * p.ldz;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int64_t col0 = v0 + c * 32;
      if (col0 >= vend) break;
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait();
      const int64_t j = yl - c * 32;
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 32; q += 2) {
        float d0 = g * ex2_approx(fmaf(as_f(r[q]), kLog2e, nl));
        float d1 = g * ex2_approx(fmaf(as_f(r[q + 1]), kLog2e, nl));
        if (q == j) d0 -= g;
        if (q + 1 == j) d1 -= g;
        w[q / 2] = pack_bf16x2(d0, d1);
      }
      if (!row_ok) continue;
      if (col0 + 32 <= vend) {
        uint4* dst = reinterpret_cast<uint4*>(out + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      } else {
        uint16_t* dst = reinterpret_cast<uint16_t*>(out + col0);
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (col0 + q < vend) dst[q] = static_cast<uint16_t>(w[q / 2] >> (16 * (q & 1)));
      }
    }
  }
};

// ------------------------------------------------------------------ store
enum StoreMode : int { kStoreF32 = 0, kAddF32 = 1, kStoreBf16AddPartial = 2, kStoreBf16 = 3 };

struct EpiStore {
  struct Params {
    void* out;              // f32 or bf16 [M][ld_out]
    const float* partial;   // f32 [M][ld_out] (mode kStoreBf16AddPartial)
    int64_t ld_out;
    int64_t M, N;           // valid rows / cols of the output
    int mode;
  };
  __device__ static void run(const Params& p, uint32_t taddr, int64_t row, int /*mb*/, int nb) {
    const int64_t n0 = static_cast<int64_t>(nb) * kBN;
    const int64_t nend = min(n0 + kBN, p.N);
    const bool row_ok = row < p.M;
    const int64_t roff = (row_ok ? row : 0) * p.ld_out;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int64_t col0 = n0 + c * 32;
      if (col0 >= nend) break;
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait();
      if (!row_ok) continue;
      const bool full = col0 + 32 <= nend;
      float v[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = as_f(r[q]);
      if (p.mode == kAddF32 || p.mode == kStoreBf16AddPartial) {
        const float* src = (p.mode == kAddF32 ? static_cast<const float*>(p.out) : p.partial) + roff + col0;
        if (full) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 a = reinterpret_cast<const float4*>(src)[q];
            v[4 * q] += a.x;
            v[4 * q + 1] += a.y;
            v[4 * q + 2] += a.z;
            v[4 * q + 3] += a.w;
          }
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q)
            if (col0 + q < nend) v[q] += src[q];
        }
      }
      if (p.mode == kStoreF32 || p.mode == kAddF32) {
        float* dst = static_cast<float*>(p.out) + roff + col0;
        if (full) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q)
            if (col0 + q < nend) dst[q] = v[q];
        }
      } else {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + roff + col0;
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) w[q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
        if (full) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q)
            if (col0 + q < nend)
              reinterpret_cast<uint16_t*>(dst)[q] = static_cast<uint16_t>(w[q / 2] >> (16 * (q & 1)));
        }
      }
    }
  }
};

// ------------------------------------------------------------------ host side
namespace {

// 2-D bf16 tensor map over a row-major [rows][cols] matrix with leading
// dimension `ld` elements; box = {box_cols (inner), box_rows}, 128B swizzle,
// out-of-bounds elements read as zero.
bool make_tmap_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <bool A_MN, bool B_MN, class Epi>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, int64_t M, int64_t Ncols, int64_t K,
                        const typename Epi::Params& ep, uint32_t* status, cudaStream_t stream, int group_m) {
  auto kern = umma_gemm_kernel<A_MN, B_MN, Epi>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kGemmSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  GemmArgs a;
  a.sched.num_m = static_cast<int>((M + kBM - 1) / kBM);
  a.sched.num_n = static_cast<int>((Ncols + kBN - 1) / kBN);
  a.sched.group_m = group_m < 1 ? 1 : group_m;
  a.num_k = static_cast<int>((K + kBK - 1) / kBK);
  a.status = status;
  const int total = a.sched.num_m * a.sched.num_n;
  const int grid = total < sm_count() ? total : sm_count();
  kern<<<grid, kGemmThreads, kGemmSmemBytes, stream>>>(ta, tb, a, ep);
  return cudaGetLastError();
}

}  // namespace

int lse_maxseg(int64_t V, int64_t Vs, int T) {
  // shard segments one 256-wide tile can touch: at most floor(255 / Vs) + 2, and at most T
  (void)V;
  int64_t m = (kBN - 1) / Vs + 2;
  if (m > T) m = T;
  return static_cast<int>(m);
}

int64_t lse_num_vtiles(int64_t V) { return (V + kBN - 1) / kBN; }

cudaError_t bf16_lse_stats(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H,
                           int64_t V, int64_t Vs, float2* partial, int maxseg, float* zy, uint32_t* status,
                           cudaStream_t stream) {
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, X, N, H, H, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, W, V, H, H, kBK, kBN)) return cudaErrorInvalidValue;
  EpiLseStats::Params p{partial, zy, targets, N, V, Vs, maxseg};
  return launch_gemm<false, false, EpiLseStats>(ta, tb, N, V, H, p, status, stream, 16);
}

cudaError_t bf16_dz_chunk(const void* X, const void* W, const int64_t* targets, const float* lse, const float* g,
                          int64_t N, int64_t H, int64_t c0, int64_t Vc, void* dz, int64_t ldz, uint32_t* status,
                          cudaStream_t stream) {
  CUtensorMap ta, tb;
  const uint8_t* Wc = static_cast<const uint8_t*>(W) + c0 * H * 2;
  if (!make_tmap_bf16(&ta, X, N, H, H, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, Wc, Vc, H, H, kBK, kBN)) return cudaErrorInvalidValue;
  EpiDZ::Params p{static_cast<__nv_bfloat16*>(dz), ldz, lse, g, targets, N, c0, Vc};
  return launch_gemm<false, false, EpiDZ>(ta, tb, N, Vc, H, p, status, stream, 16);
}

cudaError_t bf16_dx_chunk(const void* dz, int64_t ldz, const void* W, int64_t N, int64_t H, int64_t c0,
                          int64_t Vc, void* out, const float* partial, int mode, uint32_t* status,
                          cudaStream_t stream) {
  // dX[N,H] (+)= dZ_c[N,Vc] * W_c[Vc,H]: A = dZ_c (K-major), B = W_c viewed as
  // [K=Vc rows][N=H cols] (MN-major).
  CUtensorMap ta, tb;
  const uint8_t* Wc = static_cast<const uint8_t*>(W) + c0 * H * 2;
  if (!make_tmap_bf16(&ta, dz, N, Vc, ldz, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, Wc, Vc, H, H, 64, kBK)) return cudaErrorInvalidValue;
  EpiStore::Params p{out, partial, H, N, H, mode};
  return launch_gemm<false, true, EpiStore>(ta, tb, N, H, Vc, p, status, stream, 8);
}

cudaError_t bf16_dw_chunk(const void* dz, int64_t ldz, const void* X, int64_t N, int64_t H, int64_t c0,
                          int64_t Vc, float* dW, uint32_t* status, cudaStream_t stream) {
  // dW_c[Vc,H] = dZ_c^T[Vc,N] * X[N,H]: A = dZ_c viewed as [K=N rows][M=Vc cols]
  // (MN-major), B = X viewed as [K=N rows][N=H cols] (MN-major).
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, dz, N, Vc, ldz, 64, kBK)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, X, N, H, H, 64, kBK)) return cudaErrorInvalidValue;
  EpiStore::Params p{dW + c0 * H, nullptr, H, Vc, H, kStoreF32};
  return launch_gemm<true, true, EpiStore>(ta, tb, Vc, H, N, p, status, stream, 8);
}

// Plain GEMM entry used by the unit tests of the core: D[M,N] = A * B^T with
// A/B K-major or MN-major, fp32 output.
cudaError_t bf16_gemm_test(const void* A, const void* B, float* D, int64_t M, int64_t Ncols, int64_t K,
                           int a_mn, int b_mn, uint32_t* status, cudaStream_t stream) {
  CUtensorMap ta, tb;
  bool ok = a_mn ? make_tmap_bf16(&ta, A, K, M, M, 64, kBK) : make_tmap_bf16(&ta, A, M, K, K, kBK, kBM);
  ok = ok && (b_mn ? make_tmap_bf16(&tb, B, K, Ncols, Ncols, 64, kBK)
                   : make_tmap_bf16(&tb, B, Ncols, K, K, kBK, kBN));
  if (!ok) return cudaErrorInvalidValue;
  EpiStore::Params p{D, nullptr, Ncols, M, Ncols, kStoreF32};
  if (!a_mn && !b_mn) return launch_gemm<false, false, EpiStore>(ta, tb, M, Ncols, K, p, status, stream, 8);
  if (!a_mn && b_mn) return launch_gemm<false, true, EpiStore>(ta, tb, M, Ncols, K, p, status, stream, 8);
  if (a_mn && b_mn) return launch_gemm<true, true, EpiStore>(ta, tb, M, Ncols, K, p, status, stream, 8);
  return launch_gemm<true, false, EpiStore>(ta, tb, M, Ncols, K, p, status, stream, 8);
}

}  // namespace vp
