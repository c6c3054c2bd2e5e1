// The low-rank correction of a VQ3 linear layer, y_lr = U (V x') for the rotated
// input rows x', in FP32; the output step of the decode kernel and the epilogue
// of the tensor-core GEMM add it before the single FP16 rounding of y.
//
// Source: model card "anemll/anemll-forge-qwen3.8-27B", release-comparison table
// row "Token mixers" (rank-64 factors) and "ANEMLL ANE LLM conversion pipeline",
// "Facts" (rank-64 residual correction): the weight is diag(s) C[idx] + U V on
// the rotated input.
//
// Projection: one CTA computes 8 rows x 8 factor rows j over one chunk of 512
// inputs: warp w takes row r = 8 * blockIdx.z + w, each lane 8 consecutive
// inputs of each 256-input step (one 16-byte load of x' and of each of the 8 V
// rows), and the 8 sums are reduced across the warp in a fixed order. The
// chunks' sums are added in chunk order by the expansion kernel, so the result
// does not depend on timing.
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

constexpr int kChunk = 512;  // inputs per CTA of the projection

__global__ void __launch_bounds__(256) lowrank_project_kernel(const uint16_t* __restrict__ xr, int rows, int d_in,
                                                              const uint16_t* __restrict__ V, int rank,
                                                              float* __restrict__ part, int xr_mma_order) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kc = blockIdx.x;
  const int j0 = blockIdx.y * 8;
  const int r = blockIdx.z * 8 + warp;
  if (r >= rows) return;  // whole warp: no block-wide synchronisation below
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const uint16_t* xrow = xr + (size_t)r * d_in;
#pragma unroll
  for (int step = 0; step < kChunk / 256; ++step) {
    const int i0 = kc * kChunk + step * 256 + 8 * lane;
    if (i0 < d_in) {  // d_in is a multiple of 64: an 8-input group is wholly in or out
      float xv[8];
      unpack8(*reinterpret_cast<const uint4*>(xrow + i0), xv);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        float vv[8];
        if (xr_mma_order) {
          // x' holds the inputs of its 16-column group in the GEMM's operand order: take
          // the V entries of the inputs that positions i0 .. i0+7 hold
          const uint16_t* vrow = V + (size_t)(j0 + jj) * d_in + (i0 & ~15);
          float v16[16];
          unpack8(__ldg(reinterpret_cast<const uint4*>(vrow)), *reinterpret_cast<float(*)[8]>(v16));
          unpack8(__ldg(reinterpret_cast<const uint4*>(vrow + 8)), *reinterpret_cast<float(*)[8]>(v16 + 8));
#pragma unroll
          for (int k = 0; k < 8; ++k) vv[k] = v16[mma_order_input((i0 & 15) + k)];
        } else {
          unpack8(__ldg(reinterpret_cast<const uint4*>(V + (size_t)(j0 + jj) * d_in + i0)), vv);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[jj] = fmaf(vv[k], xv[k], acc[jj]);
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < 8; ++jj)
#pragma unroll
    for (int h = 16; h > 0; h >>= 1) acc[jj] += __shfl_xor_sync(0xffffffffu, acc[jj], h);
  if (lane == 0) {
    float* o = part + ((size_t)kc * rows + r) * rank + j0;  // chunk kc's sums
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) o[jj] = acc[jj];
  }
}

// y_lr[r][o] = sum_q U[o][q] z[r][q], z[r][q] = sum over chunks kc = 0, 1, ... of
// part[kc][r][q] in that order. One CTA: 256 output channels x 16 rows; z of its
// rows is summed into shared memory once, each thread keeps its U row in registers.
__global__ void __launch_bounds__(256) lowrank_expand_kernel(const float* __restrict__ part, int n_chunks, int rows,
                                                             int rank, const uint16_t* __restrict__ U, int d_out,
                                                             float* __restrict__ ylr) {
  __shared__ float zs[16][64];
  const int r0 = blockIdx.y * 16;
  for (int e = threadIdx.x; e < 16 * 64; e += blockDim.x) {
    const int rr = e / 64, q = e % 64;
    float s = 0.f;  // entries past the rank stay zero
    if (q < rank && r0 + rr < rows)
      for (int kc = 0; kc < n_chunks; ++kc) s += __ldg(part + ((size_t)kc * rows + r0 + rr) * rank + q);
    zs[rr][q] = s;
  }
  __syncthreads();
  const int o = blockIdx.x * 256 + threadIdx.x;
  if (o >= d_out) return;
  float u[64];
#pragma unroll
  for (int q8 = 0; q8 < 8; ++q8) {
    if (q8 * 8 < rank) {
      float f[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(U + (size_t)o * rank + q8 * 8)), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) u[q8 * 8 + k] = f[k];
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) u[q8 * 8 + k] = 0.f;
    }
  }
  for (int rr = 0; rr < 16 && r0 + rr < rows; ++rr) {
    float y = 0.f;
#pragma unroll
    for (int q = 0; q < 64; ++q) y = fmaf(u[q], zs[rr][q], y);  // entries past the rank are zero
    ylr[(size_t)(r0 + rr) * d_out + o] = y;
  }
}

}  // namespace

int lowrank_chunks(int d_in) { return (d_in + kChunk - 1) / kChunk; }

cudaError_t launch_lowrank(const uint16_t* xr, int rows, int d_in, const uint16_t* V, const uint16_t* U, int rank,
                           int d_out, float* part, float* ylr, cudaStream_t st, int xr_mma_order) {
  if (rows <= 0 || rank <= 0) return cudaSuccess;
  const int n_kc = lowrank_chunks(d_in);
  const dim3 g1((unsigned)n_kc, (unsigned)(rank / 8), (unsigned)((rows + 7) / 8));
  lowrank_project_kernel<<<g1, 256, 0, st>>>(xr, rows, d_in, V, rank, part, xr_mma_order);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 g2((unsigned)((d_out + 255) / 256), (unsigned)((rows + 15) / 16));
  lowrank_expand_kernel<<<g2, 256, 0, st>>>(part, n_kc, rows, rank, U, d_out, ylr);
  return cudaGetLastError();
}

}  // namespace vq3
