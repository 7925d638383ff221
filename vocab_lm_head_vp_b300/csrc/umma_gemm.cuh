// Persistent tcgen05 GEMM core for sm_103a: D[128 x 256] tiles of A * B^T with
// bf16 operands staged by TMA into 128-byte-swizzled shared memory and fp32
// accumulators in tensor memory.  The epilogue is a template parameter, so
// the same main loop serves the forward log-sum-exp statistics, the backward
// logit-gradient recompute and the dX / dW contractions.
//
// Roles (192 threads, one CTA per SM):
//   warp 0      one lane issues TMA loads into a kStages-deep ring
//   warp 1      allocates 512 TMEM columns; one lane issues tcgen05.mma
//   warps 2..5  epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, i.e. one
//               accumulator row (token / vocab row) per thread
// Two 128x256 fp32 accumulators (2 x 256 TMEM columns) let the epilogue of
// tile i overlap the MMAs of tile i+1.
//
// kMB = 2 makes each CTA tile 256 x 256: two 128-row A blocks per stage share
// the stage's B block (two MMAs per 16-deep K step, one per accumulator), so
// the CTAs running at one time cover twice the output rows per pass over B
// and B is streamed from L2 / DRAM half as often.  Both 256-column
// accumulators then belong to one tile (no overlap of epilogue and MMAs: for
// long K loops, such as dX's over the vocabulary, it does not matter) and the
// ring has 3 stages of 64 KB instead of 4 of 48 KB.
//
// Operand layouts (A is M x K, B is N x K; "MN-major" = M (or N) contiguous):
//   K-major : one TMA box {64 K, rows} per stage; swizzle atoms of 8 rows x
//             128 B stacked along the rows (stride 1024 B); the k-th 16-wide
//             slice starts 32 B further.
//   MN-major: boxes {64 MN, 64 K}; each box is 64 K-rows of 128 B, i.e. 8
//             swizzle atoms of 8 K-rows stacked along K (stride 1024 B);
//             consecutive 64-wide MN blocks are 8 KB apart; the k-th
//             16-deep slice starts 2 KB further.
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"

namespace vp {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr uint32_t kMnBoxBytes = 64 * kBK * 2;  // one {64 MN, 64 K} box: 8 KB
constexpr size_t kGemmSmemBytes = 1024 + kStages * kStageBytes + 256;

// Pipeline shape of a kernel whose CTA tile is kMB 128-row blocks by 256 columns.
template <int kMB>
struct GemmShape {
  static_assert(kMB == 1 || kMB == 2, "one or two 128-row blocks per CTA tile");
  static constexpr int kStg = kMB == 1 ? kStages : 3;    // ring stages
  static constexpr int kAcc = kMB == 1 ? 2 : 1;          // accumulator sets (2 x 256 TMEM columns in all)
  static constexpr uint32_t kAStage = kMB * kABytes;
  static constexpr uint32_t kStage = kAStage + kBBytes;
  static constexpr size_t kSmem = 1024 + kStg * kStage + 256;
};
static_assert(GemmShape<1>::kSmem == kGemmSmemBytes && GemmShape<2>::kSmem <= kGemmSmemBytes,
              "both tile shapes fit the same shared-memory budget");
// Epilogues that store through TMA stage one 32-row x 128-byte box per warp,
// double-buffered: 4 warps x 2 x 4 KB.
constexpr uint32_t kStoreBoxBytes = 32 * 128;
constexpr uint32_t kStoreStagingBytes = 4 * 2 * kStoreBoxBytes;

// Per-warp state of a TMA-storing epilogue.
struct EpiCtx {
  uint8_t* stg;     // this warp's two 4 KB staging boxes (1024-byte aligned)
  int buf;          // box to fill next
  int lane;
  int64_t row0;     // first output row of this warp's 32-row block
};

// Write this thread's 128-byte row (8 x 16 B) into the warp's staging box in
// the 128-byte swizzled order TMA expects (chunk j of row r at j ^ (r & 7)),
// then one lane stores the 32-row box at (c0, row0).  All 32 lanes call it.
__device__ __forceinline__ void stage_and_store(EpiCtx& ctx, const CUtensorMap* tm, const uint32_t (&w)[32],
                                                int32_t c0) {
  uint8_t* box = ctx.stg + ctx.buf * kStoreBoxBytes;
  if (ctx.lane == 0) bulk_wait_group_read<1>();   // the store that last used this box has read it
  __syncwarp();
  uint4* row = reinterpret_cast<uint4*>(box + ctx.lane * 128);
#pragma unroll
  for (int j = 0; j < 8; ++j) row[j ^ (ctx.lane & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (ctx.lane == 0) {
    tma_store_2d(tm, box, c0, static_cast<int32_t>(ctx.row0));
    bulk_commit_group();
  }
  ctx.buf ^= 1;
}

struct TileSched {
  int num_m, num_n, group_m;
  // Tile id -> (m block, n block): ids run down groups of `group_m` m-blocks
  // first so that CTAs working at the same time share operand tiles in L2.
  __device__ __forceinline__ void tile(int id, int& mb, int& nb) const {
    const int per_group = group_m * num_n;
    const int g = id / per_group;
    const int first_m = g * group_m;
    const int gsz = min(num_m - first_m, group_m);
    const int r = id - g * per_group;
    mb = first_m + r % gsz;
    nb = r / gsz;
  }
};

// Roles that may be told to issue nothing (a diagnostic of the bounded
// waits: the other roles' waits then run out and the CTA takes its abort path).
enum GemmHold : int { kHoldNone = 0, kHoldProducer = 1, kHoldMma = 2 };

struct GemmArgs {
  TileSched sched;
  int num_k;           // number of 64-wide K blocks
  uint32_t* status;    // device status word (VP_DEV_* bits)
  uint64_t wait_ns;    // limit of every mbarrier wait
  int hold;            // GemmHold (kHoldNone outside diagnostics)
  int64_t sk_iters;    // > 0: stream-K over tiles x num_k (tile, k-block) iterations; 0: whole tiles
};

// First stream-K iteration of CTA c out of G: floor(c * I / G), without
// forming the product c * I.
__host__ __device__ __forceinline__ int64_t sk_begin(int64_t c, int64_t G, int64_t I) {
  return c * (I / G) + (c * (I % G)) / G;
}

// A CTA's share of a launch, one piece at a time: the k-blocks [kb0, kb1) of
// one tile.  Whole tiles (blockIdx.x, + gridDim.x, ...) by default; with
// stream-K the contiguous iteration range [sk_begin(c), sk_begin(c + 1)) cut
// at tile edges, so every CTA gets the same number of k-blocks whatever the
// tile count.  A piece that is not a whole tile goes to partial slot 2c (the
// CTA's first piece) or 2c + 1 (its last); a fix-up pass adds the slots of a
// tile in CTA order, which is k order.
struct Piece {
  int tile, kb0, kb1, slot;   // slot -1: a whole tile
};
struct WorkIter {
  int64_t i, hi, first_tile;
  int tile, step, total, num_k, cta;
  bool sk;
  __device__ WorkIter(const GemmArgs& a, int total_tiles, bool none) {
    total = none ? 0 : total_tiles;
    num_k = a.num_k;
    cta = static_cast<int>(blockIdx.x);
    step = static_cast<int>(gridDim.x);
    tile = cta;
    sk = a.sk_iters > 0;
    i = sk ? sk_begin(cta, step, a.sk_iters) : 0;
    hi = (sk && !none) ? sk_begin(cta + 1, step, a.sk_iters) : 0;
    first_tile = i / num_k;
  }
  __device__ __forceinline__ bool next(Piece& p) {
    if (!sk) {
      if (tile >= total) return false;
      p.tile = tile;
      p.kb0 = 0;
      p.kb1 = num_k;
      p.slot = -1;
      tile += step;
      return true;
    }
    if (i >= hi) return false;
    const int64_t t = i / num_k;
    p.tile = static_cast<int>(t);
    p.kb0 = static_cast<int>(i - t * num_k);
    p.kb1 = static_cast<int>(min(static_cast<int64_t>(num_k), p.kb0 + (hi - i)));
    p.slot = (p.kb0 == 0 && p.kb1 == num_k) ? -1 : (t == first_tile ? 2 * cta : 2 * cta + 1);
    i += p.kb1 - p.kb0;
    return true;
  }
};

// A stream-K partial piece: this thread's accumulator row (256 fp32 columns)
// into the partial workspace row `row` through TMA (32-column boxes).
__device__ __forceinline__ void store_partial_f32(EpiCtx& ctx, const CUtensorMap* tm, uint32_t taddr) {
#pragma unroll 1
  for (int b = 0; b < kBN / 32; ++b) {
    uint32_t r[32];
    __syncwarp();
    tmem_ld32(taddr + b * 32, r);
    tmem_ld_wait();
    stage_and_store(ctx, tm, r, b * 32);
  }
}

__device__ __forceinline__ void record_failure(uint32_t* status, volatile int* abort, uint32_t bit) {
  *abort = 1;
  if (status) atomicOr(status, bit);
}

// tmP: the fp32 partial workspace of stream-K launches, rows of 256 columns,
// slot s at row s * kMB * 128 (unused when args.sk_iters == 0).
template <bool A_MN, bool B_MN, class Epi, int kMB = 1>
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
                     const GemmArgs args, const typename Epi::Params ep) {
  using S = GemmShape<kMB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;                           // kStg x kMB x 16 KB
  uint8_t* sB = smem + S::kStg * S::kAStage;    // kStg x 32 KB
  uint8_t* sC = smem + S::kStg * S::kStage;     // Epi::kStagingBytes (0 or 32 KB)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sC + Epi::kStagingBytes);
  uint64_t* full = bars;                        // TMA -> MMA
  uint64_t* empty = bars + S::kStg;             // MMA -> TMA
  uint64_t* tfull = bars + 2 * S::kStg;         // MMA -> epilogue (kAcc accumulator sets)
  uint64_t* tempty = tfull + S::kAcc;           // epilogue -> MMA
  uint64_t* drain = tempty + S::kAcc;           // MMA completion at exit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ int never_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStg; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < S::kAcc; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4 * 32);
    }
    mbar_init(drain, 1);
    *abort = 0;
    never_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (Epi::kStagingBytes) tma_prefetch_desc(&tmC);
    if (Epi::kStagingBytes && args.sk_iters > 0) tma_prefetch_desc(&tmP);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = args.sched.num_m * args.sched.num_n;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;   // bit s: stage s has a load in flight / its parity
      WorkIter it(args, total, args.hold == kHoldProducer);
      Piece pc;
      while (it.next(pc)) {
        int mb, nb;
        args.sched.tile(pc.tile, mb, nb);
        bool ok = true;
        for (int kb = pc.kb0; kb < pc.kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort, args.wait_ns)) {
            record_failure(args.status, abort, 0x1u);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], S::kStage);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          uint8_t* a = sA + stage * S::kAStage;
          uint8_t* b = sB + stage * kBBytes;
          const int k0 = kb * kBK;
#pragma unroll
          for (int h = 0; h < kMB; ++h) {
            const int m0 = (mb * kMB + h) * kBM;
            if (!A_MN) {
              tma_load_2d(a + h * kABytes, &tmA, &full[stage], k0, m0);
            } else {
              tma_load_2d(a + h * kABytes, &tmA, &full[stage], m0, k0);
              tma_load_2d(a + h * kABytes + kMnBoxBytes, &tmA, &full[stage], m0 + 64, k0);
            }
          }
          if (!B_MN) {
            tma_load_2d(b, &tmB, &full[stage], k0, nb * kBN);
          } else {
#pragma unroll
            for (int i = 0; i < kBN / 64; ++i)
              tma_load_2d(b + i * kMnBoxBytes, &tmB, &full[stage], nb * kBN + 64 * i, k0);
          }
          if (++stage == S::kStg) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Every load this thread issued must land before the CTA can exit.
      for (int s = 0; s < S::kStg; ++s)
        if (armed & (1u << s)) mbar_wait(&full[s], (armed_parity >> s) & 1u, &never_abort, args.wait_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      WorkIter it(args, total, args.hold == kHoldMma);
      Piece pc;
      while (it.next(pc)) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort, args.wait_ns)) {
          record_failure(args.status, abort, 0x2u);
          break;
        }
        tc_fence_after();
        // accumulator set acc: kMB x 256 columns (acc is always 0 when kMB = 2)
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kMB * kBN);
        bool ok = true;
        for (int kb = pc.kb0; kb < pc.kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort, args.wait_ns)) {
            record_failure(args.status, abort, 0x2u);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_addr(sA + stage * S::kAStage);
          const uint32_t b0 = smem_addr(sB + stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = B_MN ? sdesc_sw128(b0 + kk * 2048, kMnBoxBytes, 1024)
                                     : sdesc_sw128(b0 + kk * 32, 16, 1024);
#pragma unroll
            for (int h = 0; h < kMB; ++h) {
              const uint32_t ah = a0 + h * kABytes;
              const uint64_t ad = A_MN ? sdesc_sw128(ah + kk * 2048, kMnBoxBytes, 1024)
                                       : sdesc_sw128(ah + kk * 32, 16, 1024);
              umma_bf16(d_tmem + h * kBN, ad, bd, idesc, (kb != pc.kb0 || kk != 0) ? 1u : 0u);
            }
          }
          umma_commit(&empty[stage]);
          if (++stage == S::kStg) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == S::kAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued above must finish before TMEM is released.
      umma_commit(drain);
      mbar_wait(drain, 0, &never_abort, args.wait_ns);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int quad = warp & 3;
    EpiCtx ctx{sC + (warp - 2) * 2 * kStoreBoxBytes, 0, lane, 0};
    int acc = 0;
    uint32_t acc_phase = 0;
    WorkIter it(args, total, false);
    Piece pc;
    while (it.next(pc)) {
      int mb, nb;
      args.sched.tile(pc.tile, mb, nb);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort, args.wait_ns));
      if (!ok) {
        if (lane == 0) record_failure(args.status, abort, 0x4u);
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < kMB; ++h) {
        const uint32_t taddr = tmem_base + static_cast<uint32_t>((acc * kMB + h) * kBN) +
                               (static_cast<uint32_t>(quad * 32) << 16);
        if (pc.slot < 0) {
          ctx.row0 = static_cast<int64_t>(mb * kMB + h) * kBM + quad * 32;
          Epi::run(ep, &tmC, taddr, ctx.row0 + lane, nb, ctx);
        } else if constexpr (Epi::kStagingBytes > 0) {
          ctx.row0 = static_cast<int64_t>(pc.slot * kMB + h) * kBM + quad * 32;
          store_partial_f32(ctx, &tmP, taddr);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == S::kAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (Epi::kStagingBytes && lane == 0) bulk_wait_group<0>();   // this warp's stores are complete
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace vp
