// Persistent tcgen05 GEMM over CTA pairs (cta_group::2): each pair of SMs
// computes 256 x 256 tiles of A * B^T.  Each CTA stages its own 128 rows of A
// and 128 rows of B per 64-deep K block; one MMA instruction issued by the
// pair's leader reads both halves of A and of B from the two CTAs' shared
// memory, and each CTA's tensor memory receives its 128 x 256 accumulator.
// Against one 128 x 256 tile per SM this halves the B bytes every SM reads
// from L2 and from shared memory per flop.
//
// Roles per CTA (192 threads): warp 0 lane 0 issues TMA loads (both CTAs;
// completion is counted on the leader's full barrier), warp 1 allocates the
// pair's TMEM and, in the leader only, lane 0 issues the MMAs; warps 2..5 run
// the epilogue on the CTA's own accumulator rows and report back to the
// leader's tmem-empty barrier.  The epilogue classes are those of the
// one-SM kernel.
#pragma once
#include "umma_gemm.cuh"

namespace vp {

constexpr int kStages2 = 6;
constexpr uint32_t kAHalfBytes = 128 * kBK * 2;  // 16 KB: this CTA's 128 rows of A
constexpr uint32_t kBHalfBytes = 128 * kBK * 2;  // 16 KB: this CTA's 128 rows of B
constexpr uint32_t kStage2Bytes = kAHalfBytes + kBHalfBytes;
constexpr size_t kGemm2SmemBytes = 1024 + kStages2 * kStage2Bytes + 256;
constexpr int kPairBM = 256;  // tile rows per pair

template <bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const GemmArgs args,
                         const typename Epi::Params ep) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;                            // kStages2 x 16 KB
  uint8_t* sB = smem + kStages2 * kAHalfBytes;   // kStages2 x 16 KB
  uint8_t* sC = smem + kStages2 * kStage2Bytes;  // Epi::kStagingBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(sC + Epi::kStagingBytes);
  uint64_t* full = bars;                  // leader: both CTAs' TMA bytes landed
  uint64_t* empty = bars + kStages2;      // both: MMAs done reading the stage
  uint64_t* tfull = bars + 2 * kStages2;  // both: accumulator ready
  uint64_t* tempty = tfull + 2;           // leader: both CTAs' epilogues drained it
  uint64_t* drain = tempty + 2;           // leader: all MMAs complete at exit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ int never_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t half = rank & 1u;           // 0: leader of the pair
  const uint32_t leader = rank & ~1u;
  const uint16_t pair_mask = static_cast<uint16_t>(3u << leader);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * 4 * 32);
    }
    mbar_init(drain, 1);
    *abort = 0;
    never_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (Epi::kStagingBytes) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // barriers of both CTAs initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = args.sched.num_m * args.sched.num_n;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      const int first = args.hold == kHoldProducer ? total : pair;   // the diagnostic hold: issue nothing
      for (int tile = first; tile < total; tile += npairs) {
        int mb, nb;
        args.sched.tile(tile, mb, nb);
        const int m0 = mb * kPairBM + static_cast<int>(half) * 128;
        const int n0 = nb * kBN + static_cast<int>(half) * 128;
        bool ok = true;
        for (int kb = 0; kb < args.num_k; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort, args.wait_ns)) {
            record_failure(args.status, abort, 0x1u);
            ok = false;
            break;
          }
          if (half == 0) {
            mbar_arrive_expect_tx(&full[stage], 2 * kStage2Bytes);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          const uint32_t bar = map_to_rank(&full[stage], leader);
          uint8_t* a = sA + stage * kAHalfBytes;
          uint8_t* b = sB + stage * kBHalfBytes;
          const int k0 = kb * kBK;
          if (!A_MN) {
            tma_load_2d_pair(a, &tmA, bar, k0, m0);
          } else {
            tma_load_2d_pair(a, &tmA, bar, m0, k0);
            tma_load_2d_pair(a + kMnBoxBytes, &tmA, bar, m0 + 64, k0);
          }
          if (!B_MN) {
            tma_load_2d_pair(b, &tmB, bar, k0, n0);
          } else {
            tma_load_2d_pair(b, &tmB, bar, n0, k0);
            tma_load_2d_pair(b + kMnBoxBytes, &tmB, bar, n0 + 64, k0);
          }
          if (++stage == kStages2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (half == 0) {
        // Both CTAs' loads into every armed stage must land before the pair exits.
        for (int s = 0; s < kStages2; ++s)
          if (armed & (1u << s)) mbar_wait(&full[s], (armed_parity >> s) & 1u, &never_abort, args.wait_ns);
      } else if (*abort) {
        // The leader stopped consuming: give this CTA's in-flight loads time to land.
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && half == 0) {
      // ------------------------------------------------ MMA issuer (leader only)
      constexpr uint32_t idesc = idesc_bf16_f32(kPairBM, kBN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      const int first = args.hold == kHoldMma ? total : pair;   // the diagnostic hold: issue nothing
      for (int tile = first; tile < total; tile += npairs) {
        if (!mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort, args.wait_ns)) {
          record_failure(args.status, abort, 0x2u);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        bool ok = true;
        for (int kb = 0; kb < args.num_k; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort, args.wait_ns)) {
            record_failure(args.status, abort, 0x2u);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_addr(sA + stage * kAHalfBytes);
          const uint32_t b0 = smem_addr(sB + stage * kBHalfBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(a0 + kk * 2048, kMnBoxBytes, 1024)
                                     : sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b0 + kk * 2048, kMnBoxBytes, 1024)
                                     : sdesc_sw128(b0 + kk * 32, 16, 1024);
            umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair(&empty[stage], pair_mask);
          if (++stage == kStages2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[acc], pair_mask);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit_pair(drain, static_cast<uint16_t>(1u << leader));
      mbar_wait(drain, 0, &never_abort, args.wait_ns);
    }
  } else {
    // -------------------------------------------------- epilogue warps (both CTAs)
    const int quad = warp & 3;
    EpiCtx ctx{sC + (warp - 2) * 2 * kStoreBoxBytes, 0, lane, 0};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < total; tile += npairs) {
      int mb, nb;
      args.sched.tile(tile, mb, nb);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort, args.wait_ns));
      if (!ok) {
        if (lane == 0) record_failure(args.status, abort, 0x4u);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * kBN) + (static_cast<uint32_t>(quad * 32) << 16);
      ctx.row0 = static_cast<int64_t>(mb) * kPairBM + half * 128 + quad * 32;
      Epi::run(ep, &tmC, taddr, ctx.row0 + lane, nb, ctx);
      tc_fence_before();
      mbar_arrive_cluster(map_to_rank(&tempty[acc], leader));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (Epi::kStagingBytes && lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync();  // the leader's MMAs no longer read either CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace vp
