/*
 * vp_testing.h -- diagnostic entry point of libvp for checking the tcgen05
 * GEMM core on its own, apart from the cross-entropy epilogues.
 *
 * The pages define no plain GEMM; this call exists so that the tensor-core
 * main loop (TMA staging, shared-memory descriptors for K-major and MN-major
 * operands, TMEM accumulation) can be compared with a library matmul before
 * the vocab-parallel epilogues are layered on it.
 */
#ifndef VP_TESTING_H
#define VP_TESTING_H

#include "vp.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * vp_test_gemm_bf16 -- D[M,N] = A * B^T in fp32 from bf16 operands.
 *   a_mn_major == 0: A is [M,K] row-major (K contiguous)
 *   a_mn_major != 0: A is stored as [K,M] row-major (M contiguous)
 *   b_mn_major == 0: B is [N,K] row-major;  != 0: B stored as [K,N]
 *   D: f32 [M,N] row-major, overwritten.
 *   workspace: >= 16 device bytes, 16-byte aligned (device status word).
 * The contiguous dimension of each operand must be a multiple of 8 and N a
 * multiple of 4; all pointers 16-byte aligned (else VP_ERR_UNSUPPORTED).
 */
vp_status vp_test_gemm_bf16(const void* A, const void* B, float* D, int64_t M, int64_t N, int64_t K,
                            int a_mn_major, int b_mn_major, void* workspace, void* stream);

/*
 * vp_test_set_gemm_variant -- select the tcgen05 GEMM forms used by every
 * later bf16 call in this process:
 *   0 (default): the logits GEMMs on one SM per 128 x 256 tile (the epilogue
 *      overlapping the next tile's MMAs); dX on one SM per 256 x 256 or
 *      128 x 256 tile, whichever fills the waves better; dW as dW^T = X^T dZ
 *      with each 256 x 256 tile on a pair of SMs (cta_group::2);
 *   1: each 256 x 256 tile of every GEMM on a pair of SMs;
 *   2: one SM per 128 x 256 tile for every GEMM, and dW = dZ^T X directly;
 *   3: as 0, but the logits GEMMs run in clusters of two CTAs on vertically
 *      adjacent 128 x 256 tiles, each CTA loading half of the shared W tile and
 *      multicasting it into both (TMA multicast), each MMA on its own SM's
 *      shared memory; bit-identical to form 0.
 * All compute the same results within rounding; this exists to compare them.
 * Other values: VP_ERR_INVALID_ARG.
 */
vp_status vp_test_set_gemm_variant(int variant);

/*
 * vp_test_dx_plan -- how a bf16 dX GEMM (dX = dZ W, `rows` token rows, H
 * output columns) would run on a grid of `sms` persistent CTAs under the
 * current GEMM form, without launching anything (host arithmetic only):
 *   tile_rows: 256 (two 128-row A blocks per CTA sharing each W block) or 128;
 *   streamk:   1 when the launch splits tiles x K-blocks evenly over the CTAs
 *              (fewer 256-row tiles than CTAs, but at least a quarter as many,
 *              and whole waves well over the work), else 0;
 *   cost:      the relative time the plan is chosen by, in waves of 128 x 256
 *              tiles (a 256-row wave counting 2, a 128-row wave 1.15; for
 *              stream-K the 128-row tiles per CTA).
 * The fused call's default token chunk is chosen with the same costs.
 * rows, H or sms <= 0, or a null output: VP_ERR_INVALID_ARG.
 */
vp_status vp_test_dx_plan(int64_t rows, int64_t H, int sms, int32_t* tile_rows, int32_t* streamk, double* cost);

/*
 * vp_test_set_wait_fault -- exercise the bounded waits of the tcgen05 GEMMs.
 * Applies to every later bf16 GEMM launch of this process (one-SM, SM-pair and
 * multicast-cluster forms; in a pair, both CTAs' producers or the leader's MMA
 * issuer; in a multicast cluster, both CTAs' producers or MMA issuers):
 *   mode 0: normal operation (the default);
 *   mode 1: the TMA producer issues no load, so the MMA issuer's wait for
 *           data runs out (VP_DEV_TIMEOUT_MMA) and the epilogue's wait for an
 *           accumulator ends with it (VP_DEV_TIMEOUT_EPILOGUE);
 *   mode 2: the MMA issuer issues no MMA, so the producer's wait for a free
 *           stage runs out with its loads in flight (VP_DEV_TIMEOUT_PRODUCER;
 *           it first waits for those loads to land) and the epilogue's wait
 *           ends with it.
 *   wait_ns: the limit of every mbarrier wait in those launches; 0 restores
 *           the default (1 s).
 * A CTA that gives up drains what it issued, frees its tensor memory and
 * exits; the call's forward outputs (loss, lse, shard statistics) come out NaN
 * and the workspace's status word holds the bits.  Process-global, not
 * thread-safe.
 */
vp_status vp_test_set_wait_fault(int mode, uint64_t wait_ns);

/*
 * Stage timing for measurement harnesses.  While enabled, every libvp call
 * records a CUDA event on its stream before and after each kernel it
 * launches, so a harness can attribute device time to kernels inside its
 * own timed region.  Process-global, not thread-safe; meant for one
 * benchmarking thread.
 *
 * vp_stage_timing_enable(max_launches): max_launches > 0 creates the events
 *   (2 per launch) and starts recording from empty; 0 stops and frees them.
 *   Timed regions beyond max_launches are not recorded; they are counted
 *   (vp_stage_timing_dropped), so a harness can reject partial totals.
 * vp_stage_timing_read(ms, counts, n): waits for the recorded events and
 *   writes, for stage s < n, the summed milliseconds and the number of
 *   kernels launched in the stage's timed regions (embed_bwd several per
 *   region); returns the number of stages, or -1 on a
 *   CUDA error.
 * vp_stage_timing_dropped(): timed regions not recorded since the last
 *   vp_stage_timing_enable because all max_launches slots were in use.
 * vp_stage_name(s): the stage's name (static storage), NULL past the end.
 */
vp_status vp_stage_timing_enable(int max_launches);
int vp_stage_timing_read(float* ms, int32_t* counts, int n);
int vp_stage_timing_dropped(void);
const char* vp_stage_name(int stage);

#ifdef __cplusplus
}
#endif

#endif /* VP_TESTING_H */
