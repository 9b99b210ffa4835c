// fp32 64 x 64 tile products on the CUDA cores, shared by the chunk-parallel kernels (backward,
// encoder forward).  Tiles live in shared memory with a padded row stride of kLD floats.
#pragma once

#include <cuda_runtime.h>

namespace zs {
namespace tiles {

constexpr int kLD = 68;  // 16-byte aligned rows; rows 68 floats apart fall in different banks

// 64 x 64 fp32 products from shared tiles (row stride kLD = 68 floats): thread (tr = tid / 16,
// tc = tid % 16) accumulates rows tr + 16 x and columns tc + 16 y (x, y < 4) of  op(A) op(B)
// over k < 64, op(A)(r, k) = TA ? A[k][r] : A[r][k],  op(B)(k, c) = TB ? B[c][k] : B[k][c].
// Four k at a time; operands along k are read as 16-byte vectors.  The eight threads of a
// 16-byte load phase read eight rows 68 floats apart, i.e. disjoint bank quadruples.
template <bool TA, bool TB>
__device__ __forceinline__ void gemm64(const float* A, const float* B, float (&acc)[4][4]) {
  const int tr = threadIdx.x >> 4, tc = threadIdx.x & 15;
#pragma unroll 2
  for (int k0 = 0; k0 < 64; k0 += 4) {
    float av[4][4], bv[4][4];  // [k - k0][row or column index x / y]
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      if (TA) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) av[kk][x] = A[(k0 + kk) * kLD + tr + 16 * x];
      } else {
        const float4 t = *reinterpret_cast<const float4*>(A + (tr + 16 * x) * kLD + k0);
        av[0][x] = t.x; av[1][x] = t.y; av[2][x] = t.z; av[3][x] = t.w;
      }
      if (TB) {
        const float4 t = *reinterpret_cast<const float4*>(B + (tc + 16 * x) * kLD + k0);
        bv[0][x] = t.x; bv[1][x] = t.y; bv[2][x] = t.z; bv[3][x] = t.w;
      } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) bv[kk][x] = B[(k0 + kk) * kLD + tc + 16 * x];
      }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = __fmaf_rn(av[kk][x], bv[kk][y], acc[x][y]);
  }
}

__device__ __forceinline__ void zero44(float (&acc)[4][4]) {
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) acc[x][y] = 0.0f;
}

// Sum over the 16 threads of a half warp that share a row group.
__device__ __forceinline__ float sum16(float v) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}


}  // namespace tiles
}  // namespace zs
