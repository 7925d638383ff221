// Transpose of a bf16 matrix: X (or a token chunk of it) into X^T, the
// K-major A operand of the dW^T = X^T dZ GEMM.  HBM-bound.
#include <cuda_runtime.h>

#include <cstdint>

#include "vp_internal.h"

namespace vp {
namespace {

// out[c][r] = in[r][c] for a bf16 [rows][cols] matrix; cols a multiple of 8.
// 64 x 64 tiles through shared memory, 16-byte loads along the input rows and
// 16-byte stores along the output rows (8 input rows of one column) where the
// 8 rows exist and ld_out keeps the store 16-byte aligned; 2-byte stores at a
// ragged edge.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ in, int64_t rows,
                                                             int64_t cols, int64_t ld_in, uint16_t* __restrict__ out,
                                                             int64_t ld_out) {
  __shared__ uint16_t t[64][64 + 2];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64, c0 = static_cast<int64_t>(blockIdx.x) * 64;
  for (int e = threadIdx.x; e < 64 * 8; e += blockDim.x) {
    const int r = e >> 3, cv = (e & 7) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + r < rows && c0 + cv < cols) v = *reinterpret_cast<const uint4*>(in + (r0 + r) * ld_in + c0 + cv);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      t[r][cv + 2 * q] = static_cast<uint16_t>(w[q] & 0xffffu);
      t[r][cv + 2 * q + 1] = static_cast<uint16_t>(w[q] >> 16);
    }
  }
  __syncthreads();
  const bool vec_ok = (ld_out % 8) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  for (int e = threadIdx.x; e < 64 * 8; e += blockDim.x) {
    const int c = e >> 3, rv = (e & 7) * 8;   // output row c0 + c, its 8 columns from input rows r0 + rv ..
    if (c0 + c >= cols) continue;
    uint16_t* o = out + (c0 + c) * ld_out + r0 + rv;
    if (vec_ok && r0 + rv + 8 <= rows) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = static_cast<uint32_t>(t[rv + 2 * q][c]) | (static_cast<uint32_t>(t[rv + 2 * q + 1][c]) << 16);
      *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int q = 0; q < 8 && r0 + rv + q < rows; ++q) o[q] = t[rv + q][c];
    }
  }
}

}  // namespace

cudaError_t transpose_bf16(const void* in, int64_t rows, int64_t cols, int64_t ld_in, void* out, int64_t ld_out,
                           cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
  transpose_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(in), rows, cols, ld_in,
                                                  static_cast<uint16_t*>(out), ld_out);
  return cudaGetLastError();
}

}  // namespace vp
