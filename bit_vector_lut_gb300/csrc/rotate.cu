// Online Hadamard rotation and the residual/RMSNorm step.
//
// fwht_rotate: out[r, blk] = H_b diag(s_blk) x[r, blk] / sqrt(b) for every
// b-wide block of every row, H_b in Sylvester (natural) order. Source: model
// card "anemll/anemll-forge-qwen3.8-27B", section "Release 0.2: three-bit MLP,
// token-mixer rotations, distilled weights", bullet "Token-mixer rotations"
// (1,024-wide Hadamard blocks with seeded signs, the MLP inputs rotated the
// same way).
//
// One CTA owns one (row, block): each thread keeps b/128 values in registers,
// the butterflies whose partner is in the same thread run in registers, those
// across lanes use warp shuffles and those across warps go through shared
// memory. FP32 arithmetic, one FP16 rounding at the end.
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
VQ3_BOUNDS_RECORD(rotate)
namespace {

constexpr int kRotThreads = 128;

// Element j of the block lives in thread (j % 128) slot (j / 128) while the
// block is in "lane-major" form. Butterflies of stride h < 32 pair lanes within
// a warp (shuffle), strides 32 and 64 pair warps (shared memory), strides >= 128
// pair slots of the same thread (registers).
__device__ __forceinline__ float load_elem(const uint16_t* p) { return __half2float(__ushort_as_half(*p)); }
__device__ __forceinline__ float load_elem(const float* p) { return *p; }

// out[row][col] row-major FP16 (may alias an FP16 x: every element is read before
// any is written). T: FP16 (uint16_t) or FP32 input. With mma_order the columns of
// each 16-column group are stored in the tensor-core GEMM's operand order (see
// mma_order_col).
template <int B, typename T>
__global__ void __launch_bounds__(kRotThreads) fwht_kernel(const T* x, int n, const uint32_t* __restrict__ signs,
                                                            uint16_t* out, float scale, int mma_order) {
  constexpr int V = (B + kRotThreads - 1) / kRotThreads;  // values per thread
  constexpr int ACTIVE = B < kRotThreads ? B : kRotThreads;
  __shared__ float sm[V * kRotThreads];
  const int tid = threadIdx.x;
  const int blocks_per_row = n / B;
  const int row = blockIdx.x / blocks_per_row;
  const int blk = blockIdx.x % blocks_per_row;
  const size_t base = (size_t)row * n + (size_t)blk * B;

  float v[V];
#pragma unroll
  for (int s = 0; s < V; ++s) {
    const int j = s * kRotThreads + tid;
    float f = 0.f;
    if (tid < ACTIVE && VQ3_IN(base + j, (size_t)gridDim.x * B, 1)) {  // grid = rows x blocks per row
      f = load_elem(x + base + j);
      if (signs) {
        const int col = blk * B + j;
        if (VQ3_IN(col >> 5, n / 32, 2) && ((__ldg(signs + (col >> 5)) >> (col & 31)) & 1u)) f = -f;
      }
    }
    v[s] = f;
  }

  // strides 1..16 (and up to B/2 when B <= 32): lanes of one warp
#pragma unroll
  for (int h = 1; h < 32 && h < B; h <<= 1) {
#pragma unroll
    for (int s = 0; s < V; ++s) {
      const float o = __shfl_xor_sync(0xffffffffu, v[s], h);
      v[s] = (tid & h) ? (o - v[s]) : (v[s] + o);
    }
  }
  // strides 32 and 64: across warps through shared memory
#pragma unroll
  for (int h = 32; h < kRotThreads && h < B; h <<= 1) {
#pragma unroll
    for (int s = 0; s < V; ++s) sm[s * kRotThreads + tid] = v[s];
    __syncthreads();
#pragma unroll
    for (int s = 0; s < V; ++s) {
      const float o = sm[s * kRotThreads + (tid ^ h)];
      v[s] = (tid & h) ? (o - v[s]) : (v[s] + o);
    }
    __syncthreads();
  }
  // strides >= 128: slots of the same thread
#pragma unroll
  for (int hs = 1; hs < V; hs <<= 1) {
#pragma unroll
    for (int s = 0; s < V; ++s) {
      if ((s & hs) == 0) {
        const float a = v[s], c = v[s + hs];
        v[s] = a + c;
        v[s + hs] = a - c;
      }
    }
  }

  const size_t row_base = (size_t)row * n;
#pragma unroll
  for (int s = 0; s < V; ++s) {
    const int j = s * kRotThreads + tid;
    const int col = blk * B + j;
    if (tid < ACTIVE && VQ3_IN(row_base + (mma_order ? mma_order_col(col) : col), (size_t)gridDim.x * B, 3))
      out[row_base + (mma_order ? mma_order_col(col) : col)] = __half_as_ushort(__float2half_rn(v[s] * scale));
  }
}

template <int B, typename T>
cudaError_t launch_b(const T* x, int rows, int n, const uint32_t* signs, uint16_t* out, int mma_order,
                     cudaStream_t st) {
  const long long grid = (long long)rows * (n / B);
  fwht_kernel<B, T><<<(unsigned)grid, kRotThreads, 0, st>>>(x, n, signs, out, 1.0f / sqrtf((float)B), mma_order);
  return cudaGetLastError();
}

// resid_out <- fp16(resid_in + delta); normed <- fp16(resid_out * rsqrt(mean(resid_out^2) + eps))
__global__ void __launch_bounds__(256) residual_rmsnorm_kernel(const uint16_t* resid_in, const uint16_t* delta,
                                                               uint16_t* resid_out, int n, float eps,
                                                               uint16_t* normed) {
  __shared__ float red[8];
  const size_t base = (size_t)blockIdx.x * n;
  float ss = 0.f;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    float r = __half2float(__ushort_as_half(resid_in[base + j]));
    if (delta) {
      const __half s = __float2half_rn(r + __half2float(__ushort_as_half(delta[base + j])));
      resid_out[base + j] = __half_as_ushort(s);
      r = __half2float(s);
    } else if (resid_out != resid_in) {
      resid_out[base + j] = resid_in[base + j];
    }
    ss += r * r;
  }
#pragma unroll
  for (int h = 16; h > 0; h >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, h);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)n + eps);
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    // the same thread wrote resid_out[base + j] above
    const float r = __half2float(__ushort_as_half(resid_out[base + j]));
    normed[base + j] = __half_as_ushort(__float2half_rn(r * inv));
  }
}

// r_next = fp16(r + d) and, per 16 columns, the sum of r_next^2 in column order (each
// square rounded to FP32, then added): the residual step that ends one layer of the
// stack and starts the next one's RMSNorm. One CTA per row, one thread per 16 columns.
__global__ void __launch_bounds__(256) residual_add_ss_kernel(const uint16_t* __restrict__ r,
                                                              const uint16_t* __restrict__ d,
                                                              uint16_t* __restrict__ r_next, float* __restrict__ ss,
                                                              int n) {
  const size_t base = (size_t)blockIdx.x * n;
  for (int g = threadIdx.x; g < n / 16; g += blockDim.x) {
    float s = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!VQ3_IN(base + 16 * g + 8 * h + 7, (size_t)gridDim.x * n, 4)) continue;  // grid = rows
      const uint4 rv = *reinterpret_cast<const uint4*>(r + base + 16 * g + 8 * h);
      const uint4 dv = *reinterpret_cast<const uint4*>(d + base + 16 * g + 8 * h);
      const __half2* rh = reinterpret_cast<const __half2*>(&rv);
      const __half2* dh = reinterpret_cast<const __half2*>(&dv);
      uint4 ov;
      __half2* oh = reinterpret_cast<__half2*>(&ov);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 a = __half22float2(rh[k]), b = __half22float2(dh[k]);
        oh[k] = __floats2half2_rn(a.x + b.x, a.y + b.y);
        const float2 o = __half22float2(oh[k]);
        s += __fmul_rn(o.x, o.x);
        s += __fmul_rn(o.y, o.y);
      }
      *reinterpret_cast<uint4*>(r_next + base + 16 * g + 8 * h) = ov;
    }
    if (ss) ss[(size_t)blockIdx.x * (n / 16) + g] = s;
  }
}

}  // namespace

namespace {
template <typename T>
cudaError_t launch_any(const T* x, int rows, int n, int block, const uint32_t* signs, uint16_t* out, int mma_order,
                       cudaStream_t st) {
  if (mma_order && n % 16) return cudaErrorInvalidValue;
  switch (block) {
    case 2: return launch_b<2, T>(x, rows, n, signs, out, mma_order, st);
    case 4: return launch_b<4, T>(x, rows, n, signs, out, mma_order, st);
    case 8: return launch_b<8, T>(x, rows, n, signs, out, mma_order, st);
    case 16: return launch_b<16, T>(x, rows, n, signs, out, mma_order, st);
    case 32: return launch_b<32, T>(x, rows, n, signs, out, mma_order, st);
    case 64: return launch_b<64, T>(x, rows, n, signs, out, mma_order, st);
    case 128: return launch_b<128, T>(x, rows, n, signs, out, mma_order, st);
    case 256: return launch_b<256, T>(x, rows, n, signs, out, mma_order, st);
    case 512: return launch_b<512, T>(x, rows, n, signs, out, mma_order, st);
    case 1024: return launch_b<1024, T>(x, rows, n, signs, out, mma_order, st);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_fwht(const uint16_t* x, int rows, int n, int block, const uint32_t* signs,
                        uint16_t* out, cudaStream_t st, int mma_order) {
  return launch_any<uint16_t>(x, rows, n, block, signs, out, mma_order, st);
}

cudaError_t launch_fwht_f32(const float* x, int rows, int n, int block, const uint32_t* signs, uint16_t* out,
                            cudaStream_t st, int mma_order) {
  return launch_any<float>(x, rows, n, block, signs, out, mma_order, st);
}

cudaError_t launch_residual_rmsnorm(uint16_t* resid, const uint16_t* delta, int rows, int n, float eps,
                                    uint16_t* normed, cudaStream_t st) {
  residual_rmsnorm_kernel<<<rows, 256, 0, st>>>(resid, delta, resid, n, eps, normed);
  return cudaGetLastError();
}

cudaError_t launch_residual_add_ss(const uint16_t* r, const uint16_t* d, uint16_t* r_next, float* ss, int rows,
                                   int n, cudaStream_t st) {
  residual_add_ss_kernel<<<rows, 256, 0, st>>>(r, d, r_next, ss, n);
  return cudaGetLastError();
}

cudaError_t launch_residual_rmsnorm2(const uint16_t* resid_in, const uint16_t* delta, uint16_t* resid_out, int rows,
                                     int n, float eps, uint16_t* normed, cudaStream_t st) {
  residual_rmsnorm_kernel<<<rows, 256, 0, st>>>(resid_in, delta, resid_out, n, eps, normed);
  return cudaGetLastError();
}

}  // namespace vq3
