// The low-rank correction of a VQ3 linear layer at prefill sizes (17 rows and more),
// y_lr = U (V x') for the rotated input rows x', in FP32; the epilogue of the tensor-core
// GEMM adds it before the single FP16 rounding of y. (Below 17 rows the decode kernel forms
// the same correction itself.)
//
// Source: model card "anemll/anemll-forge-qwen3.8-27B", release-comparison table
// row "Token mixers" (rank-64 factors) and "ANEMLL ANE LLM conversion pipeline",
// "Facts" (rank-64 residual correction): the weight is diag(s) C[idx] + U V on
// the rotated input.
//
// Three launches, all on m16n8k16 tensor cores or plain adds:
//   projection  part[sp] = x' V^T over input split sp (64-row tiles x the 64 factor rows,
//               x' and V staged by 16-byte cp.async, two stages);
//   reduction   z = sum of part[sp] in split order (FP32);
//   expansion   y_lr = z U^T (64-row x 128-output tiles; z enters the MMA as two FP16
//               parts hi = fp16(z), lo = fp16(z - hi), U as FP16).
// The split count grows as the row tiles shrink, so that a few rows still fill the GPU.
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
VQ3_BOUNDS_RECORD(lowrank)
namespace {

constexpr int kLT = 64;        // rows per tile
constexpr int kLK = 64;        // inputs per stage
constexpr int kLS = kLK + 8;   // staged row stride in halves: 4 words past a multiple of 32

__device__ __forceinline__ void mma_lr(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src) : "memory");
}
__device__ __forceinline__ void zero16(void* dst) { *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u); }
__device__ __forceinline__ uint32_t ld32(const uint16_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// Input pair held by position pair p of a 16-input group when x' is in the GEMM's operand
// order (positions 2p, 2p+1 hold inputs 2c, 2c+1 with c = p/2 + 4 (p % 2)).
__device__ __forceinline__ int held_pair(int p) { return (p >> 1) + 4 * (p & 1); }

// part[sp][r][q] = sum over the inputs of split sp of x'[r][i] V[q][i]. CTA (row tile, split):
// warp w takes rows 16w .. 16w+15 of the tile and all 64 factor rows (8 n-tiles).
template <bool kMmaOrder>
__global__ void __launch_bounds__(128) lowrank_project_kernel(const uint16_t* __restrict__ xr, int rows, int d_in,
                                                              const uint16_t* __restrict__ V, int rank,
                                                              float* __restrict__ part, int n_split) {
  __shared__ __align__(16) uint16_t xs[2][kLT * kLS];
  __shared__ __align__(16) uint16_t vs[2][64 * kLS];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int r0 = blockIdx.x * kLT, sp = blockIdx.y;
  const int n_kg = d_in / kLK;
  const int kg0 = (int)((long long)sp * n_kg / n_split), kg1 = (int)((long long)(sp + 1) * n_kg / n_split);
  auto stage = [&](int buf, int kg) {
    for (int i = tid; i < 64 * 8; i += 128) {
      const int row = i >> 3, c = i & 7;
      uint16_t* dx = xs[buf] + row * kLS + c * 8;
      if (r0 + row < rows && VQ3_IN((size_t)(r0 + row) * d_in + (size_t)kg * kLK + c * 8 + 7, (size_t)rows * d_in, 1))
        cp16(dx, xr + (size_t)(r0 + row) * d_in + (size_t)kg * kLK + c * 8);
      else zero16(dx);
      uint16_t* dv = vs[buf] + row * kLS + c * 8;
      if (row < rank && VQ3_IN((size_t)row * d_in + (size_t)kg * kLK + c * 8 + 7, (size_t)rank * d_in, 2))
        cp16(dv, V + (size_t)row * d_in + (size_t)kg * kLK + c * 8);
      else zero16(dv);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  float acc[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[n][j] = 0.f;
  // the V word offsets of b0 / b1 within a 16-input group (the inputs x' holds at positions 2t.. / 2t+8..)
  const int vo0 = kMmaOrder ? 2 * held_pair(t) : 2 * t, vo1 = kMmaOrder ? 2 * held_pair(t + 4) : 2 * t + 8;
  if (kg0 < kg1) stage(0, kg0);
  for (int kg = kg0; kg < kg1; ++kg) {
    const int buf = (kg - kg0) & 1;
    if (kg + 1 < kg1) {
      stage(buf ^ 1, kg + 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();  // the stage's copies (and zero fills) of every thread are visible
    const uint16_t* xa = xs[buf] + (16 * warp + g) * kLS + 2 * t;
    const uint16_t* vb = vs[buf] + g * kLS;
#pragma unroll
    for (int s = 0; s < kLK / 16; ++s) {
      const uint32_t a[4] = {ld32(xa + 16 * s), ld32(xa + 8 * kLS + 16 * s), ld32(xa + 16 * s + 8),
                             ld32(xa + 8 * kLS + 16 * s + 8)};
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const uint16_t* vr = vb + 8 * n * kLS + 16 * s;
        mma_lr(acc[n], a, ld32(vr + vo0), ld32(vr + vo1));
      }
    }
    __syncthreads();  // every warp is done with this stage before it is refilled
  }
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const int q = 8 * n + 2 * t;
    if (q >= rank) continue;  // rank is a multiple of 8: q and q + 1 are both in or both out
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = r0 + 16 * warp + g + 8 * h;
      if (r < rows && VQ3_IN(((size_t)sp * rows + r) * rank + q + 1, (size_t)n_split * rows * rank, 3))
        *reinterpret_cast<float2*>(part + ((size_t)sp * rows + r) * rank + q) = make_float2(acc[n][2 * h], acc[n][2 * h + 1]);
    }
  }
}

// z[r][q] = part[0][r][q] + part[1][r][q] + ... in split order.
__global__ void __launch_bounds__(256) lowrank_reduce_kernel(const float* __restrict__ part, int n_split, int n,
                                                             float* __restrict__ z) {
  const int e = blockIdx.x * 256 + threadIdx.x;
  if (e >= n) return;
  float s = 0.f;
  for (int k0 = 0; k0 < n_split; k0 += 16) {  // sixteen splits' loads in flight, added in order
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
      v[k] = k0 + k < n_split && VQ3_IN((size_t)(k0 + k) * n + e, (size_t)n_split * n, 4) ? __ldg(part + (size_t)(k0 + k) * n + e)
                                                                                          : 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) s += v[k];
  }
  z[e] = s;
}

// y_lr[r][o] = sum_q z[r][q] U[o][q]. CTA: 64 rows x 128 outputs; warp w: rows 16w .. 16w+15,
// 16 n-tiles of 8 outputs. z (FP32) enters as FP16 hi and lo parts, two MMAs per tile and k-step.
__global__ void __launch_bounds__(128) lowrank_expand_kernel(const float* __restrict__ z, int rows, int rank,
                                                             const uint16_t* __restrict__ U, int d_out,
                                                             float* __restrict__ ylr) {
  __shared__ uint32_t zh[kLT][36], zl[kLT][36];        // FP16 pairs of z [row][q pair], stride 36 words
  __shared__ __align__(16) uint16_t us[128 * kLS];    // U rows of the tile's outputs, q 0 .. 63
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int o0 = blockIdx.x * 128, r0 = blockIdx.y * kLT;
  for (int i = tid; i < 128 * 8; i += 128) {  // U: 16-byte chunks of each row (q past the rank zero)
    const int row = i >> 3, c = i & 7;
    uint16_t* du = us + row * kLS + c * 8;
    if (o0 + row < d_out && c * 8 < rank && VQ3_IN((size_t)(o0 + row) * rank + c * 8 + 7, (size_t)d_out * rank, 5))
      cp16(du, U + (size_t)(o0 + row) * rank + c * 8);
    else zero16(du);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  {
    // z pairs, split into FP16 hi / lo: the thread's 16 pairs are loaded first, then converted
    constexpr int kPer = kLT * 32 / 128;
    float2 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + 128 * k, row = i >> 5, qp = i & 31;
      v[k] = (r0 + row < rows && 2 * qp < rank && VQ3_IN((size_t)(r0 + row) * rank + 2 * qp + 1, (size_t)rows * rank, 6))
                 ? *reinterpret_cast<const float2*>(z + (size_t)(r0 + row) * rank + 2 * qp)
                                                : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + 128 * k, row = i >> 5, qp = i & 31;
      const __half2 h = __floats2half2_rn(v[k].x, v[k].y);
      const float2 e = __half22float2(h);
      const __half2 l = __floats2half2_rn(v[k].x - e.x, v[k].y - e.y);
      zh[row][qp] = *reinterpret_cast<const uint32_t*>(&h);
      zl[row][qp] = *reinterpret_cast<const uint32_t*>(&l);
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  float acc[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[n][j] = 0.f;
  const int ra = 16 * warp + g;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t ah[4] = {zh[ra][8 * s + t], zh[ra + 8][8 * s + t], zh[ra][8 * s + 4 + t], zh[ra + 8][8 * s + 4 + t]};
    const uint32_t al[4] = {zl[ra][8 * s + t], zl[ra + 8][8 * s + t], zl[ra][8 * s + 4 + t], zl[ra + 8][8 * s + 4 + t]};
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const uint16_t* ub = us + (8 * n + g) * kLS + 16 * s + 2 * t;
      const uint32_t b0 = ld32(ub), b1 = ld32(ub + 8);
      mma_lr(acc[n], ah, b0, b1);
      mma_lr(acc[n], al, b0, b1);
    }
  }
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int o = o0 + 8 * n + 2 * t;
    if (o >= d_out) continue;  // d_out is a multiple of 64: a tile's n-tiles past it are whole
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = r0 + ra + 8 * h;
      if (r < rows && VQ3_IN((size_t)r * d_out + o + 1, (size_t)rows * d_out, 7))
        *reinterpret_cast<float2*>(ylr + (size_t)r * d_out + o) = make_float2(acc[n][2 * h], acc[n][2 * h + 1]);
    }
  }
}

}  // namespace

int lowrank_chunks(int d_in, int rows) {
  // splits of the input: about two CTAs per SM over the row tiles, at most one per 64 inputs
  // and at most 32 (the reduction adds them 16 at a time)
  const int tiles = (rows + kLT - 1) / kLT;
  int n = (2 * device_sm_count() + tiles - 1) / tiles;
  const int n_kg = d_in / kLK;
  if (n > n_kg) n = n_kg;
  if (n > 32) n = 32;
  return n < 1 ? 1 : n;
}

size_t lowrank_part_floats(int d_in, int rows, int rank) {
  return ((size_t)lowrank_chunks(d_in, rows) + 1) * rows * rank;  // the splits' parts, then z
}

cudaError_t launch_lowrank(const uint16_t* xr, int rows, int d_in, const uint16_t* V, const uint16_t* U, int rank,
                           int d_out, float* part, float* ylr, cudaStream_t st, int xr_mma_order) {
  if (rows <= 0 || rank <= 0) return cudaSuccess;
  const int n_split = lowrank_chunks(d_in, rows);
  const dim3 g1((unsigned)((rows + kLT - 1) / kLT), (unsigned)n_split);
  if (xr_mma_order)
    lowrank_project_kernel<true><<<g1, 128, 0, st>>>(xr, rows, d_in, V, rank, part, n_split);
  else
    lowrank_project_kernel<false><<<g1, 128, 0, st>>>(xr, rows, d_in, V, rank, part, n_split);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  float* z = part + (size_t)n_split * rows * rank;
  const int n = rows * rank;
  lowrank_reduce_kernel<<<(n + 255) / 256, 256, 0, st>>>(part, n_split, n, z);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const dim3 g3((unsigned)((d_out + 127) / 128), (unsigned)((rows + kLT - 1) / kLT));
  lowrank_expand_kernel<<<g3, 128, 0, st>>>(z, rows, rank, U, d_out, ylr);
  return cudaGetLastError();
}

}  // namespace vq3
