// Persistent tcgen05 GEMM over clusters of two CTAs that share the B operand
// by TMA multicast: the two CTAs compute vertically adjacent 128 x 256 tiles
// (the same 256 B rows, 128 A rows each) with one-SM MMAs (cta_group::1) on
// their own shared memory, but each loads only half of the stage's B block
// and multicasts it into both CTAs.  Against one 128 x 256 tile per SM this
// halves the B bytes each SM asks of L2 per flop, without the SM-pair MMA's
// reads of the other SM's shared memory.  K-major A and B.
//
// A stage of a CTA is refilled only after both CTAs' MMAs have read it (the
// other CTA writes half of it): each MMA commit arrives on the empty barrier
// of both CTAs (count 2).  Each CTA arms its own full barrier with all of the
// stage's bytes, its own loads and the other CTA's multicast half.  Roles,
// accumulators and epilogues are those of the one-SM kernel; both CTAs walk
// the same tile sequence, so their stages and phases stay paired.
#pragma once
#include "umma_gemm_2sm.cuh"

namespace vp {

template <class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_gemm_mc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmArgs args,
                        const typename Epi::Params ep) {
  using S = GemmShape<1>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;                         // kStg x 16 KB
  uint8_t* sB = smem + S::kStg * kABytes;     // kStg x 32 KB (two 16 KB halves, one from each CTA)
  uint8_t* sC = smem + S::kStg * S::kStage;   // Epi::kStagingBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(sC + Epi::kStagingBytes);
  uint64_t* full = bars;                      // this CTA's loads + the other CTA's B half
  uint64_t* empty = bars + S::kStg;           // both CTAs' MMAs done reading the stage
  uint64_t* tfull = bars + 2 * S::kStg;
  uint64_t* tempty = tfull + S::kAcc;
  uint64_t* drain = tempty + S::kAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ int never_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t half = cluster_ctarank() & 1u;
  const uint16_t both = 3u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStg; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
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
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // both CTAs' barriers initialised before any multicast or remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = args.sched.num_m * args.sched.num_n;   // tiles of 256 rows: one per cluster
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      const int first = args.hold == kHoldProducer ? total : pair;
      for (int tile = first; tile < total; tile += npairs) {
        int mb, nb;
        args.sched.tile(tile, mb, nb);
        const int m0 = mb * kPairBM + static_cast<int>(half) * kBM;
        const int n0 = nb * kBN + static_cast<int>(half) * (kBN / 2);
        bool ok = true;
        for (int kb = 0; kb < args.num_k; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort, args.wait_ns)) {
            record_failure(args.status, abort, 0x1u);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], S::kStage);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          const int k0 = kb * kBK;
          tma_load_2d(sA + stage * kABytes, &tmA, &full[stage], k0, m0);
          tma_load_2d_multicast(sB + stage * kBBytes + half * (kBBytes / 2), &tmB, &full[stage], k0, n0, both);
          if (++stage == S::kStg) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Every stage this CTA armed must land (its loads and the other CTA's
      // half) before the cluster can exit.
      for (int s = 0; s < S::kStg; ++s)
        if (armed & (1u << s)) mbar_wait(&full[s], (armed_parity >> s) & 1u, &never_abort, args.wait_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer (each CTA)
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      const int first = args.hold == kHoldMma ? total : pair;
      for (int tile = first; tile < total; tile += npairs) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort, args.wait_ns)) {
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
          const uint32_t a0 = smem_addr(sA + stage * kABytes);
          const uint32_t b0 = smem_addr(sB + stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(d_tmem, sdesc_sw128(a0 + kk * 32, 16, 1024), sdesc_sw128(b0 + kk * 32, 16, 1024), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          umma_commit_multicast(&empty[stage], both);
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
      umma_commit(drain);
      mbar_wait(drain, 0, &never_abort, args.wait_ns);
    }
  } else {
    // -------------------------------------------------- epilogue warps
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
      ctx.row0 = static_cast<int64_t>(mb) * kPairBM + half * kBM + quad * 32;
      Epi::run(ep, &tmC, taddr, ctx.row0 + lane, nb, ctx);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == S::kAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (Epi::kStagingBytes && lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync();  // the other CTA no longer multicasts into this one or arrives on its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace vp
