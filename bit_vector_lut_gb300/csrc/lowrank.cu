// First half of the low-rank correction of a VQ3 linear layer: z = V x' for
// the rotated input rows x' (the second half, U z, is added in the output step
// of the decode kernel and in the epilogue of the tensor-core GEMM, before the
// single FP16 rounding of y).
//
// Source: model card "anemll/anemll-forge-qwen3.8-27B", release-comparison table
// row "Token mixers" (rank-64 factors) and "ANEMLL ANE LLM conversion pipeline",
// "Facts" (rank-64 residual correction): the weight is diag(s) C[idx] + U V on
// the rotated input.
//
// One CTA computes 8 rows x 8 factor rows j: warp w takes row r = 8 * blockIdx.x
// + w, each lane 8 consecutive inputs of every 256-input step (one 16-byte load
// of x' and of each of the 8 V rows), and the 8 sums are reduced across the warp
// in a fixed order (deterministic).
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 p = __half22float2(h[k]);
    f[2 * k] = p.x;
    f[2 * k + 1] = p.y;
  }
}

__global__ void __launch_bounds__(256) lowrank_project_kernel(const uint16_t* __restrict__ xr, int rows, int d_in,
                                                              const uint16_t* __restrict__ V, int rank,
                                                              float* __restrict__ z) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  const int j0 = blockIdx.y * 8;
  if (r >= rows) return;  // whole warp: no block-wide synchronisation below
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const uint16_t* xrow = xr + (size_t)r * d_in;
  for (int i0 = 8 * lane; i0 < d_in; i0 += 256) {
    float xv[8];
    unpack8(*reinterpret_cast<const uint4*>(xrow + i0), xv);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      float vv[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(V + (size_t)(j0 + jj) * d_in + i0)), vv);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[jj] = fmaf(vv[k], xv[k], acc[jj]);
    }
  }
#pragma unroll
  for (int jj = 0; jj < 8; ++jj)
#pragma unroll
    for (int h = 16; h > 0; h >>= 1) acc[jj] += __shfl_xor_sync(0xffffffffu, acc[jj], h);
  if (lane == 0) {
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) z[(size_t)r * rank + j0 + jj] = acc[jj];
  }
}

}  // namespace

cudaError_t launch_lowrank_project(const uint16_t* xr, int rows, int d_in, const uint16_t* V, int rank, float* z,
                                   cudaStream_t st) {
  if (rows <= 0 || rank <= 0) return cudaSuccess;
  const dim3 grid((unsigned)((rows + 7) / 8), (unsigned)(rank / 8));
  lowrank_project_kernel<<<grid, 256, 0, st>>>(xr, rows, d_in, V, rank, z);
  return cudaGetLastError();
}

}  // namespace vq3
