// bf16 tensor-core path of the fused LM head + vocab-parallel cross-entropy:
// the three epilogues that ride on the tcgen05 GEMM core and their launchers.
//
//   EpiLseStats  forward: per token row and per shard segment of a 256-wide
//                vocab tile, the local max m and R = sum exp(z - m) over the
//                segment's logits except one maximal one (S = 1 + R, kept
//                apart from the 1 so that a tiny R survives), plus the
//                target logit when the tile owns the target ("Vocab
//                Parallelism" sec. 5.3.1; interview note figure 2).
//   EpiLseStatsP the same statistics, plus the tile's probabilities relative
//                to its row maximum, kept in fp16 for the fused backward (the
//                saved-probability backward of sec. 5.3.2).
//   EpiDZ        backward: recomputed logits -> dZ = g (exp(z - lse) - 1[j=y])
//                stored as bf16 for one vocab chunk (sec. 5.3.2).
//   EpiStore     dX / dW: fp32 accumulator -> fp32 store, fp32 read-add-store,
//                or bf16 store (optionally adding an fp32 partial first).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "umma_gemm.cuh"
#include "umma_gemm_2sm.cuh"
#include "umma_gemm_mc.cuh"
#include "vp_internal.h"

namespace vp {

constexpr float kLog2e = 1.4426950408889634f;

// Rows (of the output's M dimension) per tile group of each launch: the
// persistent CTAs walk down a group's m-blocks before moving along n, so CTAs
// running at the same time share operand tiles in L2.
#ifndef VP_GROUP_ROWS_LOGITS
#define VP_GROUP_ROWS_LOGITS 4096   // forward / recompute: token rows (W re-read once per group)
#endif
#ifndef VP_GROUP_ROWS_LOGITS_MAX
#define VP_GROUP_ROWS_LOGITS_MAX 6144   // up to this many token rows form a single group
#endif
#ifndef VP_GROUP_ROWS_DX
#define VP_GROUP_ROWS_DX 1024       // dX: token rows
#endif
#ifndef VP_GROUP_ROWS_DW
#define VP_GROUP_ROWS_DW 2048       // dW: vocab rows
#endif

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ forward
// kStoreP = false: statistics only (the split forward; logits never stored).
// kStoreP = true (the fused forward + backward): the epilogue also writes
// p = exp(z - m_tile) in fp16 through TMA, where m_tile is the row's maximum
// over the tile's valid columns (stored in tmax).  Both forms take the same
// branches and sums, so their statistics are bit-identical.  p lies in (0, 1], where fp16
// carries 11 significant bits, so the later gradient
// exp(z - lse) = p * exp(m_tile - lse) keeps a relative error near 2^-11.
template <bool kStoreP>
struct EpiLseStatsT {
  static constexpr uint32_t kStagingBytes = kStoreP ? kStoreStagingBytes : 0;
  struct Params {
    float2* partial;          // [num_vtiles * maxseg][N] (m, R), R = S - 1
    float* zy;                // [N] target logit, written by the owning tile
    const int64_t* targets;   // [N]
    int64_t N, V, Vs;         // tokens, vocab, shard width V/T
    int maxseg;               // record slots per vocab tile
    float* tmax;              // [num_vtiles][N] row maximum of each tile (kStoreP)
    int64_t y_off;            // vocab id of W's first row (targets are ids of the whole vocabulary)
  };
  // A tile of 256 valid columns inside one shard (all but the tiles holding a
  // shard edge or the vocabulary's end): one pass for the row maximum m over
  // the tile, then one exp per logit, e = exp(z - m), stored as p = e in fp16
  // with kStoreP and summed into the tile's single (m, R) record.  Logits
  // equal to m are counted instead of summed: R = (sum over z < m) + (ties - 1).
  __device__ static void run_whole(const Params& p, const CUtensorMap* tm, uint32_t taddr, int64_t n, int nb,
                                   int64_t v0, int64_t yl, bool row_ok, EpiCtx& ctx) {
    float mx = -INFINITY, zyv = 0.f;
    bool have_zy = false;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait();
      const int64_t j = yl - c * 32;
      if (j >= 0 && j < 32) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < 32; ++q) v = (q == j) ? as_f(r[q]) : v;
        zyv = v;
        have_zy = true;
      }
      float cm = as_f(r[0]);
#pragma unroll
      for (int q = 1; q < 32; ++q) cm = fmaxf(cm, as_f(r[q]));
      mx = fmaxf(mx, cm);
    }
    const float nt = -mx * kLog2e;
    const bool warp_live = ctx.row0 < p.N;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int ties = 0;
#pragma unroll 1
    for (int b = 0; b < kBN / 64; ++b) {
      uint32_t w[kStoreP ? 32 : 1];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + b * 64 + h * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float e0 = ex2_approx(fmaf(as_f(r[q + 0]), kLog2e, nt));
          const float e1 = ex2_approx(fmaf(as_f(r[q + 1]), kLog2e, nt));
          const float e2 = ex2_approx(fmaf(as_f(r[q + 2]), kLog2e, nt));
          const float e3 = ex2_approx(fmaf(as_f(r[q + 3]), kLog2e, nt));
          const bool t0 = as_f(r[q + 0]) == mx, t1 = as_f(r[q + 1]) == mx;
          const bool t2 = as_f(r[q + 2]) == mx, t3 = as_f(r[q + 3]) == mx;
          a0 += t0 ? 0.f : e0;
          a1 += t1 ? 0.f : e1;
          a2 += t2 ? 0.f : e2;
          a3 += t3 ? 0.f : e3;
          ties += (t0 + t1) + (t2 + t3);
          if constexpr (kStoreP) {
            w[h * 16 + q / 2] = pack_f16x2(e0, e1);
            w[h * 16 + q / 2 + 1] = pack_f16x2(e2, e3);
          }
        }
      }
      // rows >= N are clipped by the tensor map
      if constexpr (kStoreP) {
        if (warp_live) stage_and_store(ctx, tm, w, static_cast<int32_t>(v0 + b * 64));
      }
    }
    if (row_ok) {
      // ties >= 1 (m is one of the logits); further ties are whole terms exp(0) = 1
      p.partial[(static_cast<int64_t>(nb) * p.maxseg) * p.N + n] =
          make_float2(mx, ((a0 + a1) + (a2 + a3)) + static_cast<float>(ties - 1));
      if (have_zy) p.zy[n] = zyv;
      if constexpr (kStoreP) p.tmax[static_cast<int64_t>(nb) * p.N + n] = mx;
    }
  }

  __device__ static void run(const Params& p, const CUtensorMap* tm, uint32_t taddr, int64_t n, int nb,
                             EpiCtx& ctx) {
    const int64_t v0 = static_cast<int64_t>(nb) * kBN;
    const int64_t vend = min(v0 + kBN, p.V);
    const bool row_ok = n < p.N;
    const int64_t yl = row_ok ? p.targets[n] - p.y_off - v0 : -1;
    int64_t t = v0 / p.Vs;
    int64_t seg_end = min((t + 1) * p.Vs, vend);
    if (vend - v0 == kBN && seg_end == vend) {
      run_whole(p, tm, taddr, n, nb, v0, yl, row_ok, ctx);
      return;
    }
    int k = 0;
    float m = -INFINITY, s = 0.f, zyv = 0.f, tmx = -INFINITY;
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
        if (kStoreP) tmx = fmaxf(tmx, cm);
        // a new maximum turns the old one into an ordinary term, and one of
        // this chunk's logits equal to it is the segment's excluded maximum
        int skip = 0;
        if (cm > m) {
          s = (s + 1.f) * ex2_approx((m - cm) * kLog2e);
          m = cm;
          skip = 1;
        }
        const float mL = m * kLog2e;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        int ties = 0;
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const bool t0 = as_f(r[q + 0]) == m, t1 = as_f(r[q + 1]) == m;
          const bool t2 = as_f(r[q + 2]) == m, t3 = as_f(r[q + 3]) == m;
          a0 += t0 ? 0.f : ex2_approx(fmaf(as_f(r[q + 0]), kLog2e, -mL));
          a1 += t1 ? 0.f : ex2_approx(fmaf(as_f(r[q + 1]), kLog2e, -mL));
          a2 += t2 ? 0.f : ex2_approx(fmaf(as_f(r[q + 2]), kLog2e, -mL));
          a3 += t3 ? 0.f : ex2_approx(fmaf(as_f(r[q + 3]), kLog2e, -mL));
          ties += (t0 + t1) + (t2 + t3);
        }
        s += ((a0 + a1) + (a2 + a3)) + static_cast<float>(ties - skip);
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
          if (kStoreP) tmx = fmaxf(tmx, z);
          if (z > m) {
            s = (s + 1.f) * ex2_approx((m - z) * kLog2e);   // the old maximum joins the sum
            m = z;
          } else {
            s += ex2_approx((z - m) * kLog2e);   // a tie adds exp(0) = 1
          }
        }
      }
    }
    if (row_ok) {
      rec[static_cast<int64_t>(k) * p.N] = make_float2(m, s);
      if (have_zy) p.zy[n] = zyv;
    }
    if constexpr (kStoreP) {
      if (row_ok) p.tmax[static_cast<int64_t>(nb) * p.N + n] = tmx;
      const bool warp_live = ctx.row0 < p.N;
      const float nt = -tmx * kLog2e;
#pragma unroll 1
      for (int b = 0; b < kBN / 64; ++b) {
        const int64_t col0 = v0 + b * 64;
        if (col0 >= vend) break;
        uint32_t w[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
          __syncwarp();
          tmem_ld32(taddr + b * 64 + h * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; q += 2)
            w[h * 16 + q / 2] = pack_f16x2(ex2_approx(fmaf(as_f(r[q]), kLog2e, nt)),
                                           ex2_approx(fmaf(as_f(r[q + 1]), kLog2e, nt)));
        }
        // columns >= V and rows >= N are clipped by the tensor map
        if (warp_live) stage_and_store(ctx, tm, w, static_cast<int32_t>(col0));
      }
    }
  }
};
using EpiLseStats = EpiLseStatsT<false>;
using EpiLseStatsP = EpiLseStatsT<true>;

// ------------------------------------------------------------------ backward dZ
// dZ boxes of 32 rows x 64 bf16 columns go out through TMA (the tensor map
// clips rows >= N and columns >= Vc).
struct EpiDZ {
  static constexpr uint32_t kStagingBytes = kStoreStagingBytes;
  struct Params {
    const float* lse;         // [N]
    const float* g;           // [N] upstream scale (0 for ignored rows)
    const int64_t* targets;   // [N]
    int64_t N;
    int64_t c0, Vc;           // chunk start (vocab id of the chunk's first column) and width
  };
  __device__ static void run(const Params& p, const CUtensorMap* tm, uint32_t taddr, int64_t n, int nb,
                             EpiCtx& ctx) {
    const int64_t v0 = static_cast<int64_t>(nb) * kBN;   // chunk-local
    const int64_t vend = min(v0 + kBN, p.Vc);
    const bool row_ok = n < p.N;
    const bool warp_live = ctx.row0 < p.N;
    const float g = row_ok ? p.g[n] : 0.f;
    const float nl = row_ok ? -p.lse[n] * kLog2e : 0.f;
    const int64_t yl = (row_ok ? p.targets[n] : -1) - p.c0 - v0;
#pragma unroll 1
    for (int b = 0; b < kBN / 64; ++b) {
      const int64_t col0 = v0 + b * 64;
      if (col0 >= vend) break;
      uint32_t w[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + b * 64 + h * 32, r);
        tmem_ld_wait();
        const int64_t j = yl - (b * 64 + h * 32);
#pragma unroll
        for (int q = 0; q < 32; q += 2) {
          float d0 = g * ex2_approx(fmaf(as_f(r[q]), kLog2e, nl));
          float d1 = g * ex2_approx(fmaf(as_f(r[q + 1]), kLog2e, nl));
          if (q == j) d0 -= g;
          if (q + 1 == j) d1 -= g;
          w[h * 16 + q / 2] = pack_bf16x2(d0, d1);
        }
      }
      if (warp_live) stage_and_store(ctx, tm, w, static_cast<int32_t>(col0));
    }
  }
};

// ------------------------------------------------------------------ store
enum StoreMode : int { kStoreF32 = 0, kAddF32 = 1, kStoreBf16AddPartial = 2, kStoreBf16 = 3 };

// fp32 modes store 32-column boxes, bf16 modes 64-column boxes, through TMA.
struct EpiStore {
  static constexpr uint32_t kStagingBytes = kStoreStagingBytes;
  struct Params {
    const float* partial;   // f32 [M][ld] read and added first (modes kAddF32, kStoreBf16AddPartial)
    int64_t ld;             // leading dimension of `partial`
    int64_t M, N;           // valid rows / cols of the output
    int mode;
  };
  __device__ static void run(const Params& p, const CUtensorMap* tm, uint32_t taddr, int64_t row, int nb,
                             EpiCtx& ctx) {
    const int64_t n0 = static_cast<int64_t>(nb) * kBN;
    const int64_t nend = min(n0 + kBN, p.N);
    const bool row_ok = row < p.M;
    const bool warp_live = ctx.row0 < p.M;
    const bool add = p.mode == kAddF32 || p.mode == kStoreBf16AddPartial;
    const float* src = add && row_ok ? p.partial + row * p.ld : nullptr;
    if (p.mode == kStoreF32 || p.mode == kAddF32) {
#pragma unroll 1
      for (int b = 0; b < kBN / 32; ++b) {
        const int64_t col0 = n0 + b * 32;
        if (col0 >= nend) break;
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + b * 32, r);
        tmem_ld_wait();
        if (src) add_partial(r, src + col0, nend - col0);
        if (warp_live) stage_and_store(ctx, tm, r, static_cast<int32_t>(col0));
      }
    } else {
#pragma unroll 1
      for (int b = 0; b < kBN / 64; ++b) {
        const int64_t col0 = n0 + b * 64;
        if (col0 >= nend) break;
        uint32_t w[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
          __syncwarp();
          tmem_ld32(taddr + b * 64 + h * 32, r);
          tmem_ld_wait();
          if (src) add_partial(r, src + col0 + h * 32, nend - col0 - h * 32);
#pragma unroll
          for (int q = 0; q < 16; ++q) w[h * 16 + q] = pack_bf16x2(as_f(r[2 * q]), as_f(r[2 * q + 1]));
        }
        if (warp_live) stage_and_store(ctx, tm, w, static_cast<int32_t>(col0));
      }
    }
  }
  // r[q] += src[q] for the q < valid columns of this 32-column slice
  __device__ static void add_partial(uint32_t (&r)[32], const float* src, int64_t valid) {
    if (valid >= 32) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 a = reinterpret_cast<const float4*>(src)[q];
        r[4 * q] = __float_as_uint(as_f(r[4 * q]) + a.x);
        r[4 * q + 1] = __float_as_uint(as_f(r[4 * q + 1]) + a.y);
        r[4 * q + 2] = __float_as_uint(as_f(r[4 * q + 2]) + a.z);
        r[4 * q + 3] = __float_as_uint(as_f(r[4 * q + 3]) + a.w);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 32; ++q)
        if (q < valid) r[q] = __float_as_uint(as_f(r[q]) + src[q]);
    }
  }
};

// dW through its transpose: the GEMM computes tiles of dW^T = X^T dZ (rows =
// hidden index h, columns = vocab index v) from K-major X^T and MN-major dZ,
// and the epilogue writes each 32 x 32 block transposed into dW [V, H] fp32
// through shared memory, adding the old values first when accumulating (the
// sum over token chunks).  A K-major A operand keeps the tensor pipe busier
// than the MN-major dZ^T that dW = dZ^T X would take as A.
struct EpiStoreT {
  static constexpr uint32_t kStagingBytes = kStoreStagingBytes;
  struct Params {
    float* out;       // dW rows of this launch's vocab range, [V][ld]
    int64_t ld;       // row length of out (H)
    int64_t V, H;     // valid vocab rows / hidden columns
    int add;          // 1: out += tile, 0: out = tile
  };
  __device__ static void run(const Params& p, const CUtensorMap* tm, uint32_t taddr, int64_t h, int nb,
                             EpiCtx& ctx) {
    (void)h;
    const int64_t h0 = ctx.row0;   // this warp's first hidden index (warp-uniform)
    if (h0 >= p.H) return;
    const int64_t vbase = static_cast<int64_t>(nb) * kBN;
    const int lane = ctx.lane;
#pragma unroll 1
    for (int b = 0; b < kBN / 32; ++b) {
      const int64_t v0 = vbase + b * 32;
      if (v0 >= p.V) break;   // uniform over the CTA
      // accumulating: lane l fetches old row v0 + l, columns h0 .. h0+31, as 8
      // 16-byte vectors (8 rows' lines in flight per load, like a row-major tile)
      float4 old[8];
      const int64_t vr = v0 + lane;
      if (p.add) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          old[q] = (vr < p.V && h0 + 4 * q < p.H)
                       ? *reinterpret_cast<const float4*>(p.out + vr * p.ld + h0 + 4 * q)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(taddr + b * 32, r);
      tmem_ld_wait();
      // the 32 x 32 block transposed into the staging box (row = vocab row), the
      // old values added row by row, then one TMA store; columns >= H and rows
      // >= V are clipped by the tensor map
      uint8_t* box = ctx.stg + ctx.buf * kStoreBoxBytes;
      if (lane == 0) bulk_wait_group_read<1>();   // the store that last used this box has read it
      __syncwarp();
      const int chunk = lane >> 2, within = (lane & 3) * 4;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        *reinterpret_cast<uint32_t*>(box + j * 128 + ((chunk ^ (j & 7)) << 4) + within) = r[j];
      if (p.add) {
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4* cell = reinterpret_cast<float4*>(box + lane * 128 + ((q ^ (lane & 7)) << 4));
          const float4 a = *cell;
          *cell = make_float4(a.x + old[q].x, a.y + old[q].y, a.z + old[q].z, a.w + old[q].w);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tm, box, static_cast<int32_t>(h0), static_cast<int32_t>(v0));
        bulk_commit_group();
      }
      ctx.buf ^= 1;
    }
  }
};

// ------------------------------------------------------------------ host side
namespace {

// Token rows per tile group of a logits GEMM over N rows: all of them when
// they are few enough that X stays in L2 beside the W tiles in use (W then
// streams from DRAM once), else VP_GROUP_ROWS_LOGITS.  A token chunk of the
// fused call (e.g. 4608 rows) would otherwise end in a small group that
// streams all of W again for a few rows.
int logits_group_rows(int64_t N) {
  return N <= VP_GROUP_ROWS_LOGITS_MAX ? static_cast<int>(N) : VP_GROUP_ROWS_LOGITS;
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix with leading
// dimension `ld` elements; box = {box_cols (inner), box_rows}, 128B swizzle,
// out-of-bounds elements read as zero.
bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int64_t rows, int64_t cols,
               int64_t ld, int box_cols, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
bool make_tmap_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows) {
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, ld, box_cols, box_rows);
}
// Output maps of the TMA-storing epilogues: boxes of 32 rows x 128 bytes.
bool make_store_tmap(CUtensorMap* m, bool bf16, const void* base, int64_t rows, int64_t cols, int64_t ld) {
  return bf16 ? make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, ld, 64, 32)
              : make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, rows, cols, ld, 32, 32);
}

// Launch-configuration facts are cached per device: a process may drive
// several GPUs, and a function's shared-memory opt-in is made per device.
constexpr int kMaxDevices = 64;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  const int dev = current_device();
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Opt `kern` in to `smem` bytes of dynamic shared memory on the current device, once.
template <class Kern>
cudaError_t ensure_smem(Kern kern, size_t smem, std::atomic<int>* done) {
  const int dev = current_device();
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
  return e;
}

// Stream-K launches use at most this many CTAs (the partial workspace holds
// two 256 x 256 fp32 slots per CTA: sk_workspace_bytes()).
constexpr int kSkMaxCtas = 160;
// The fix-up pass adds at most this many pieces (CTAs) per tile, in this many
// row slabs per tile (blocks).
constexpr int kSkMaxPieces = 8;
constexpr int kSkSlabs = 16;

// The largest number of CTAs whose stream-K iteration ranges meet one tile's
// k-blocks, for `tiles` tiles of num_k k-blocks split over G CTAs.
int sk_max_pieces(int64_t tiles, int64_t num_k, int64_t G) {
  const int64_t I = tiles * num_k;
  int64_t most = 0, c = 0;
  for (int64_t t = 0; t < tiles; ++t) {
    const int64_t lo = t * num_k, hi = lo + num_k;
    while (sk_begin(c + 1, G, I) <= lo) ++c;   // c holds iteration lo
    int64_t d = c;
    while (d + 1 < G && sk_begin(d + 1, G, I) < hi) ++d;
    if (d - c + 1 > most) most = d - c + 1;
  }
  return static_cast<int>(most);
}

// Diagnostic of the bounded waits (vp_test_set_wait_fault): a role of every
// later GEMM launch that issues nothing, and the waits' time limit.
int g_hold = kHoldNone;
uint64_t g_wait_ns = kWaitTimeoutNs;

// Stream-K plan of one launch: the partial workspace and its tensor map.
struct StreamK {
  float* ws = nullptr;    // 2 * kSkMaxCtas * 256 rows x 256 fp32 (partial slots)
  CUtensorMap tp;         // over ws, 32-row x 32-column fp32 boxes
  int64_t iters = 0;      // 0: whole tiles
  int grid = 0;
};

// kMB 128-row blocks per CTA tile (1: 128 x 256 tiles, 2: 256 x 256 tiles);
// group_m_rows: output rows per tile group.  With sk_ws, a launch whose tiles
// do not fill whole waves of the persistent grid runs stream-K (the CTAs
// split the (tile, k-block) iterations evenly) and `sk` returns the plan the
// fix-up pass needs.
template <bool A_MN, bool B_MN, class Epi, int kMB = 1>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, int64_t M,
                        int64_t Ncols, int64_t K, const typename Epi::Params& ep, uint32_t* status,
                        cudaStream_t stream, int group_m_rows, float* sk_ws = nullptr, StreamK* sk = nullptr) {
  auto kern = umma_gemm_kernel<A_MN, B_MN, Epi, kMB>;
  constexpr size_t smem = GemmShape<kMB>::kSmem + Epi::kStagingBytes;
  static std::atomic<int> attr_done[kMaxDevices];
  const cudaError_t e = ensure_smem(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  GemmArgs a;
  a.sched.num_m = static_cast<int>((M + kMB * kBM - 1) / (kMB * kBM));
  a.sched.num_n = static_cast<int>((Ncols + kBN - 1) / kBN);
  const int group_m = (group_m_rows + kMB * kBM - 1) / (kMB * kBM);
  a.sched.group_m = group_m < 1 ? 1 : group_m;
  a.num_k = static_cast<int>((K + kBK - 1) / kBK);
  a.status = status;
  a.wait_ns = g_wait_ns;
  a.hold = g_hold;
  a.sk_iters = 0;
  const int total = a.sched.num_m * a.sched.num_n;
  int grid = total < sm_count() ? total : sm_count();
  const CUtensorMap* tp = &tc;
  if (sk) sk->iters = 0;
  if (sk && sk_ws && Epi::kStagingBytes > 0) {
    const int G = sm_count() < kSkMaxCtas ? sm_count() : kSkMaxCtas;
    const int64_t iters = static_cast<int64_t>(total) * a.num_k;
    // only while no tile's k-blocks spread over more CTAs than the fix-up adds
    if (total % G != 0 && a.num_k >= 2 && iters >= G && sk_max_pieces(total, a.num_k, G) <= kSkMaxPieces) {
      sk->ws = sk_ws;
      const int64_t rows = static_cast<int64_t>(2 * G) * kMB * kBM;
      if (!make_tmap(&sk->tp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, sk_ws, rows, kBN, kBN, 32, 32))
        return cudaErrorInvalidValue;
      sk->iters = iters;
      sk->grid = G;
      a.sk_iters = iters;
      grid = G;
      tp = &sk->tp;
    }
  }
  kern<<<grid, kGemmThreads, smem, stream>>>(ta, tb, tc, *tp, a, ep);
  return cudaGetLastError();
}

// One 256 x 256 tile per CTA pair (cluster of 2) on the persistent grid of
// as many pairs as can be resident at once.
template <bool A_MN, bool B_MN, class Epi>
cudaError_t launch_gemm_2sm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, int64_t M,
                            int64_t Ncols, int64_t K, const typename Epi::Params& ep, uint32_t* status,
                            cudaStream_t stream, int group_m) {
  auto kern = umma_gemm_2sm_kernel<A_MN, B_MN, Epi>;
  constexpr size_t smem = kGemm2SmemBytes + Epi::kStagingBytes;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static std::atomic<int> attr_done[kMaxDevices];
  static std::atomic<int> pairs_cache[kMaxDevices];
  const cudaError_t e = ensure_smem(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  const int dev = current_device();
  int max_pairs = pairs_cache[dev].load(std::memory_order_relaxed);
  if (max_pairs == 0) {
    cfg.gridDim = dim3(2 * (sm_count() / 2));
    if (cudaOccupancyMaxActiveClusters(&max_pairs, kern, &cfg) != cudaSuccess || max_pairs <= 0) {
      cudaGetLastError();
      max_pairs = sm_count() / 2;
    }
    pairs_cache[dev].store(max_pairs, std::memory_order_relaxed);
  }
  GemmArgs a;
  a.sched.num_m = static_cast<int>((M + kPairBM - 1) / kPairBM);
  a.sched.num_n = static_cast<int>((Ncols + kBN - 1) / kBN);
  a.sched.group_m = group_m < 1 ? 1 : group_m;
  a.num_k = static_cast<int>((K + kBK - 1) / kBK);
  a.status = status;
  a.wait_ns = g_wait_ns;
  a.hold = g_hold;
  a.sk_iters = 0;
  const int total = a.sched.num_m * a.sched.num_n;
  const int pairs = total < max_pairs ? total : max_pairs;
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, a, ep);
}

// One 128 x 256 tile per SM, the two CTAs of a cluster on vertically adjacent
// tiles that share B by multicast (umma_gemm_mc_kernel).  K-major operands.
template <class Epi>
cudaError_t launch_gemm_mc(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, int64_t M,
                           int64_t Ncols, int64_t K, const typename Epi::Params& ep, uint32_t* status,
                           cudaStream_t stream, int group_m) {
  auto kern = umma_gemm_mc_kernel<Epi>;
  constexpr size_t smem = GemmShape<1>::kSmem + Epi::kStagingBytes;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static std::atomic<int> attr_done[kMaxDevices];
  static std::atomic<int> pairs_cache[kMaxDevices];
  const cudaError_t e = ensure_smem(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  const int dev = current_device();
  int max_pairs = pairs_cache[dev].load(std::memory_order_relaxed);
  if (max_pairs == 0) {
    cfg.gridDim = dim3(2 * (sm_count() / 2));
    if (cudaOccupancyMaxActiveClusters(&max_pairs, kern, &cfg) != cudaSuccess || max_pairs <= 0) {
      cudaGetLastError();
      max_pairs = sm_count() / 2;
    }
    pairs_cache[dev].store(max_pairs, std::memory_order_relaxed);
  }
  GemmArgs a;
  a.sched.num_m = static_cast<int>((M + kPairBM - 1) / kPairBM);
  a.sched.num_n = static_cast<int>((Ncols + kBN - 1) / kBN);
  a.sched.group_m = group_m < 1 ? 1 : group_m;
  a.num_k = static_cast<int>((K + kBK - 1) / kBK);
  a.status = status;
  a.wait_ns = g_wait_ns;
  a.hold = g_hold;
  a.sk_iters = 0;
  const int total = a.sched.num_m * a.sched.num_n;
  const int pairs = total < max_pairs ? total : max_pairs;
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, a, ep);
}

// GEMM form (vp_test_set_gemm_variant): 0 (default) one SM per tile for the
// logits and dX (dX tiles by dx_plan), dW^T on SM pairs; 1 SM pairs
// (cta_group::2, 256 x 256 tiles) everywhere; 2 one SM per 128 x 256 tile
// everywhere, dW in the direct form.
int g_variant = 0;
bool pair_kernels() { return g_variant == 1; }
// Form 3: as form 0, the logits GEMMs in multicast clusters (launch_gemm_mc).
bool logits_multicast() { return g_variant == 3; }

// B operand K-major box rows: 256 for one SM, 128 (its half) for a CTA pair.
int kmajor_b_box_rows() { return pair_kernels() ? 128 : kBN; }

template <bool A_MN, bool B_MN, class Epi, int kMB = 1>
cudaError_t launch_any(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, int64_t M,
                       int64_t Ncols, int64_t K, const typename Epi::Params& ep, uint32_t* status,
                       cudaStream_t stream, int group_m_rows, float* sk_ws = nullptr, StreamK* sk = nullptr) {
  if (sk) sk->iters = 0;
  if (pair_kernels())
    return launch_gemm_2sm<A_MN, B_MN, Epi>(ta, tb, tc, M, Ncols, K, ep, status, stream,
                                            (group_m_rows + kPairBM - 1) / kPairBM);
  if (kMB == 2 && g_variant == 2)
    return launch_gemm<A_MN, B_MN, Epi, 1>(ta, tb, tc, M, Ncols, K, ep, status, stream, group_m_rows);
  return launch_gemm<A_MN, B_MN, Epi, kMB>(ta, tb, tc, M, Ncols, K, ep, status, stream, group_m_rows, sk_ws, sk);
}

// Stream-K fix-up: blockIdx.x runs over the CTA boundaries of the launch; a
// boundary that falls inside a tile, and is that tile's first, finishes the
// tile, one slab of tile_rows / gridDim.y rows per blockIdx.y (so that the
// few split tiles still spread over the SMs).  The tile's pieces, in CTA order
// (k order), are added in fp32 and the sum finished as the store epilogue
// would: fp32 store, fp32 add onto the output, or bf16 (after adding
// `partial`).  Columns come in fours (H is a multiple of 8).
__global__ void __launch_bounds__(256) sk_fixup_kernel(const float* __restrict__ ws, int64_t iters, int G, int num_k,
                                                       TileSched sched, int tile_rows, void* __restrict__ out,
                                                       const float* __restrict__ partial, int64_t ld, int64_t M,
                                                       int64_t Ncols, int mode) {
  const int c = static_cast<int>(blockIdx.x) + 1;
  const int slab_rows = tile_rows / static_cast<int>(gridDim.y);
  const int r_begin = static_cast<int>(blockIdx.y) * slab_rows;
  const int64_t b = sk_begin(c, G, iters);
  if (b % num_k == 0) return;                                        // a tile edge: nothing split here
  const int64_t t = b / num_k;
  if (sk_begin(c - 1, G, iters) > t * num_k) return;                 // an earlier boundary inside t does it
  int c_last = c;
  while (c_last + 1 < G && sk_begin(c_last + 1, G, iters) < (t + 1) * num_k) ++c_last;
  int slots[kSkMaxPieces];
  int np = 0;
  for (int q = c - 1; q <= c_last && np < kSkMaxPieces; ++q)
    slots[np++] = (sk_begin(q, G, iters) / num_k == t) ? 2 * q : 2 * q + 1;
  int mb, nb;
  sched.tile(static_cast<int>(t), mb, nb);
  const int64_t row0 = static_cast<int64_t>(mb) * tile_rows, col0 = static_cast<int64_t>(nb) * kBN;
  for (int e = threadIdx.x; e < slab_rows * (kBN / 4); e += blockDim.x) {
    const int r = r_begin + e / (kBN / 4), cq = (e % (kBN / 4)) * 4;
    const int64_t row = row0 + r, col = col0 + cq;
    if (row >= M || col >= Ncols) continue;
    float4 acc = *reinterpret_cast<const float4*>(ws + (static_cast<int64_t>(slots[0]) * tile_rows + r) * kBN + cq);
    for (int q = 1; q < np; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(ws + (static_cast<int64_t>(slots[q]) * tile_rows + r) * kBN + cq);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int64_t o = row * ld + col;
    if (mode == kStoreF32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + o) = acc;
    } else if (mode == kAddF32) {
      float4* d = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
      const float4 x = *d;
      *d = make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
    } else {
      if (mode == kStoreBf16AddPartial) {
        const float4 x = *reinterpret_cast<const float4*>(partial + o);
        acc = make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
      }
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + o) =
          make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  }
}

}  // namespace

void set_gemm_variant(int variant) { g_variant = (variant >= 1 && variant <= 3) ? variant : 0; }

bool dw_through_xt() { return g_variant != 2; }

// Relative time of a dX launch over `rows` token rows in units of one wave of
// 128 x 256 tiles: its waves on the persistent grid, a 256-row wave counting
// twice, a 128-row wave 15% more than half of that.  Unthrottled a 128-row
// wave costs about 4% more (it streams W twice as often per row); under the
// GPU's power cap the fused step measured fastest with 15%, which also moves
// its token chunks (V = 128256: 4608 rows, not 4736).  The tile shape with
// the lower cost is taken.  (256 x 256 tiles on SM pairs, which fill waves of
// 74 pairs, were measured slower for this contraction than either one-SM form
// at equal wave counts.)
DxPlan dx_plan(int64_t rows, int64_t H) { return dx_plan_on(rows, H, sm_count()); }

DxPlan dx_plan_on(int64_t rows, int64_t H, int64_t G) {
  const int64_t cols = (H + kBN - 1) / kBN;
  const auto waves = [&](int64_t tile_rows) { return ((rows + tile_rows - 1) / tile_rows * cols + G - 1) / G; };
  const double c1 = 1.15 * static_cast<double>(waves(kBM)), c2 = 2.0 * static_cast<double>(waves(2 * kBM));
  DxPlan p;
  const bool two = g_variant != 2 && c2 <= c1;
  p.rows = two ? 2 * kBM : kBM;
  p.cost = two ? c2 : c1;
  // fewer 256-row tiles than SMs (but at least a quarter as many: with fewer,
  // the fp32 partials of tiles split over many CTAs cost more than the idle
  // SMs, measured on the MiniMind dX shape), and whole waves would take over a
  // third longer than the work: split the tiles over the SMs
  const int64_t t2 = (rows + 2 * kBM - 1) / (2 * kBM) * cols;
  const double ideal = static_cast<double>((rows + kBM - 1) / kBM * cols) / static_cast<double>(G);
  p.streamk = g_variant != 2 && 4 * t2 >= G && t2 < G && ideal < 0.75 * p.cost;
  if (p.streamk) {
    p.rows = 2 * kBM;
    p.cost = ideal;
  }
  return p;
}

size_t sk_workspace_bytes() { return size_t(2) * kSkMaxCtas * 2 * kBM * kBN * sizeof(float); }

void set_wait_fault(int hold, uint64_t wait_ns) {
  g_hold = (hold == kHoldProducer || hold == kHoldMma) ? hold : kHoldNone;
  g_wait_ns = wait_ns > 0 ? wait_ns : kWaitTimeoutNs;
}

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
                           cudaStream_t stream, int64_t y_off) {
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, X, N, H, H, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, W, V, H, H, kBK, logits_multicast() ? 128 : kmajor_b_box_rows()))
    return cudaErrorInvalidValue;
  EpiLseStats::Params p{partial, zy, targets, N, V, Vs, maxseg, nullptr, y_off};
  if (logits_multicast())
    return launch_gemm_mc<EpiLseStats>(ta, tb, ta, N, V, H, p, status, stream,
                                       (logits_group_rows(N) + kPairBM - 1) / kPairBM);
  return launch_any<false, false, EpiLseStats>(ta, tb, ta, N, V, H, p, status, stream, logits_group_rows(N));
}

cudaError_t bf16_lse_stats_p(const void* X, const void* W, const int64_t* targets, int64_t N, int64_t H, int64_t V,
                             int64_t Vs, float2* partial, int maxseg, float* zy, float* tmax, void* P, int64_t ldp,
                             uint32_t* status, cudaStream_t stream) {
  CUtensorMap ta, tb, tc;
  if (!make_tmap_bf16(&ta, X, N, H, H, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, W, V, H, H, kBK, logits_multicast() ? 128 : kmajor_b_box_rows()))
    return cudaErrorInvalidValue;
  // fp16 boxes of 32 rows x 64 columns (128 bytes), clipped at V columns and N rows
  if (!make_tmap(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, P, N, V, ldp, 64, 32)) return cudaErrorInvalidValue;
  EpiLseStatsP::Params p{partial, zy, targets, N, V, Vs, maxseg, tmax, 0};
  if (logits_multicast())
    return launch_gemm_mc<EpiLseStatsP>(ta, tb, tc, N, V, H, p, status, stream,
                                        (logits_group_rows(N) + kPairBM - 1) / kPairBM);
  return launch_any<false, false, EpiLseStatsP>(ta, tb, tc, N, V, H, p, status, stream, logits_group_rows(N));
}

cudaError_t bf16_dz_chunk(const void* X, const void* W, const int64_t* targets, const float* lse, const float* g,
                          int64_t N, int64_t H, int64_t c0, int64_t Vc, void* dz, int64_t ldz, uint32_t* status,
                          cudaStream_t stream, int64_t y_off) {
  CUtensorMap ta, tb, tc;
  const uint8_t* Wc = static_cast<const uint8_t*>(W) + c0 * H * 2;
  if (!make_tmap_bf16(&ta, X, N, H, H, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, Wc, Vc, H, H, kBK, logits_multicast() ? 128 : kmajor_b_box_rows()))
    return cudaErrorInvalidValue;
  if (!make_store_tmap(&tc, true, dz, N, Vc, ldz)) return cudaErrorInvalidValue;
  EpiDZ::Params p{lse, g, targets, N, y_off + c0, Vc};
  if (logits_multicast())
    return launch_gemm_mc<EpiDZ>(ta, tb, tc, N, Vc, H, p, status, stream,
                                 (logits_group_rows(N) + kPairBM - 1) / kPairBM);
  return launch_any<false, false, EpiDZ>(ta, tb, tc, N, Vc, H, p, status, stream, logits_group_rows(N));
}

cudaError_t bf16_dx_chunk(const void* dz, int64_t ldz, const void* W, int64_t N, int64_t H, int64_t c0,
                          int64_t Vc, void* out, const float* partial, int mode, uint32_t* status,
                          cudaStream_t stream, float* sk_ws, int* kernels) {
  // dX[N,H] (+)= dZ_c[N,Vc] * W_c[Vc,H]: A = dZ_c (K-major), B = W_c viewed as
  // [K=Vc rows][N=H cols] (MN-major).
  CUtensorMap ta, tb, tc;
  const uint8_t* Wc = static_cast<const uint8_t*>(W) + c0 * H * 2;
  if (!make_tmap_bf16(&ta, dz, N, Vc, ldz, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, Wc, Vc, H, H, 64, kBK)) return cudaErrorInvalidValue;
  if (!make_store_tmap(&tc, mode >= kStoreBf16AddPartial, out, N, H, H)) return cudaErrorInvalidValue;
  EpiStore::Params p{mode == kAddF32 ? static_cast<const float*>(out) : partial, H, N, H, mode};
  // 256-row tiles stream W half as often; 128-row tiles when they fill the
  // grid's waves better (dx_plan).  Stream-K only for launches with too few
  // tiles to fill a wave: its CTAs sit at different K offsets, so they share
  // no W slices in L2, which costs more than a partly empty last wave of a
  // large launch (measured at V = 151936: 42% slower).
  StreamK sk;
  if (kernels) *kernels = 1;
  const DxPlan plan = dx_plan(N, H);
  cudaError_t e;
  if (plan.rows == 2 * kBM)
    e = launch_any<false, true, EpiStore, 2>(ta, tb, tc, N, H, Vc, p, status, stream, VP_GROUP_ROWS_DX,
                                             plan.streamk ? sk_ws : nullptr, &sk);
  else
    e = launch_any<false, true, EpiStore, 1>(ta, tb, tc, N, H, Vc, p, status, stream, VP_GROUP_ROWS_DX);
  if (e != cudaSuccess || sk.iters == 0) return e;
  if (kernels) *kernels = 2;
  TileSched sched;
  sched.num_m = static_cast<int>((N + 2 * kBM - 1) / (2 * kBM));
  sched.num_n = static_cast<int>((H + kBN - 1) / kBN);
  const int group_m = VP_GROUP_ROWS_DX / (2 * kBM);
  sched.group_m = group_m < 1 ? 1 : group_m;
  sk_fixup_kernel<<<dim3(static_cast<unsigned>(sk.grid - 1), kSkSlabs), 256, 0, stream>>>(
      sk.ws, sk.iters, sk.grid, static_cast<int>((Vc + kBK - 1) / kBK), sched, 2 * kBM, out,
      mode == kAddF32 ? static_cast<const float*>(out) : partial, H, N, H, mode);
  return cudaGetLastError();
}

cudaError_t bf16_dw_chunk(const void* dz, int64_t ldz, const void* X, int64_t N, int64_t H, int64_t c0,
                          int64_t Vc, float* dW, bool accumulate, uint32_t* status, cudaStream_t stream) {
  // dW_c[Vc,H] = dZ_c^T[Vc,N] * X[N,H]: A = dZ_c viewed as [K=N rows][M=Vc cols]
  // (MN-major), B = X viewed as [K=N rows][N=H cols] (MN-major).
  CUtensorMap ta, tb, tc;
  if (!make_tmap_bf16(&ta, dz, N, Vc, ldz, 64, kBK)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, X, N, H, H, 64, kBK)) return cudaErrorInvalidValue;
  // accumulate: dW_c += dZ_c^T X (the sum over token chunks), read and written by the same CTA
  float* out = dW + c0 * H;
  if (!make_store_tmap(&tc, false, out, Vc, H, H)) return cudaErrorInvalidValue;
  EpiStore::Params p{accumulate ? out : nullptr, H, Vc, H, accumulate ? kAddF32 : kStoreF32};
  return launch_any<true, true, EpiStore>(ta, tb, tc, Vc, H, N, p, status, stream, VP_GROUP_ROWS_DW);
}

cudaError_t bf16_dwt_chunk(const void* Xt, int64_t ldxt, const void* dz, int64_t ldz, int64_t N, int64_t H,
                           int64_t c0, int64_t Vc, float* dW, bool accumulate, uint32_t* status, cudaStream_t stream) {
  if (g_variant == 2)   // the direct form, dW = dZ^T X with both operands MN-major (for comparison)
    return cudaErrorNotSupported;
  // dW_c^T[H, Vc] = X^T[H, N] dZ_c[N, Vc]: A = X^T (K-major, K = tokens), B = dZ_c viewed as
  // [K = N rows][N = Vc cols] (MN-major); the epilogue stores each block transposed into dW.
  CUtensorMap ta, tb, tc;
  if (!make_tmap_bf16(&ta, Xt, H, N, ldxt, kBK, kBM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, dz, N, Vc, ldz, 64, kBK)) return cudaErrorInvalidValue;
  float* out = dW + c0 * H;
  if (!make_store_tmap(&tc, false, out, Vc, H, H)) return cudaErrorInvalidValue;
  EpiStoreT::Params p{out, H, Vc, H, accumulate ? 1 : 0};
  // 256 x 256 tiles on SM pairs (each SM holds half of the dZ block): measured faster for this
  // contraction than one SM per 128 x 256 tile (V128k fused step, same box: dW 13.2 vs 14.4 ms).
  // All of H's row blocks per group: consecutive tiles share one dZ column block in L2.
  return launch_gemm_2sm<false, true, EpiStoreT>(ta, tb, tc, H, Vc, N, p, status, stream,
                                                 static_cast<int>(H) / kPairBM);
}

// Plain GEMM entry used by the unit tests of the core: D[M,N] = A * B^T with
// A/B K-major or MN-major, fp32 output.
cudaError_t bf16_gemm_test(const void* A, const void* B, float* D, int64_t M, int64_t Ncols, int64_t K,
                           int a_mn, int b_mn, uint32_t* status, cudaStream_t stream) {
  CUtensorMap ta, tb, tc;
  bool ok = a_mn ? make_tmap_bf16(&ta, A, K, M, M, 64, kBK) : make_tmap_bf16(&ta, A, M, K, K, kBK, kBM);
  ok = ok && (b_mn ? make_tmap_bf16(&tb, B, K, Ncols, Ncols, 64, kBK)
                   : make_tmap_bf16(&tb, B, Ncols, K, K, kBK, kmajor_b_box_rows()));
  ok = ok && make_store_tmap(&tc, false, D, M, Ncols, Ncols);
  if (!ok) return cudaErrorInvalidValue;
  EpiStore::Params p{nullptr, Ncols, M, Ncols, kStoreF32};
  if (!a_mn && !b_mn) return launch_any<false, false, EpiStore>(ta, tb, tc, M, Ncols, K, p, status, stream, 1024);
  if (!a_mn && b_mn) return launch_any<false, true, EpiStore>(ta, tb, tc, M, Ncols, K, p, status, stream, 1024);
  if (a_mn && b_mn) return launch_any<true, true, EpiStore>(ta, tb, tc, M, Ncols, K, p, status, stream, 1024);
  return launch_any<true, false, EpiStore>(ta, tb, tc, M, Ncols, K, p, status, stream, 1024);
}

}  // namespace vp
