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

#ifdef __cplusplus
}
#endif

#endif /* VP_TESTING_H */
