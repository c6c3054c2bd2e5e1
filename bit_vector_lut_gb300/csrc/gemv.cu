// Split-K VQ3 GEMM for small row counts (weight streaming), FP32 accumulation on
// the tensor cores (m16n8k16, FP16 operands).
//
// Computes, for one or two matrices sharing a rotated input x' (gate and up):
//   y[r][o] = scale[o] * sum_i C[idx[o/2][i]][o%2] * x'[r][i]
// Weights are the MMA A operand (16 output channels x 16 inputs), the rows of
// x' are the B operand (N = 8 rows per n-tile). The per-output-channel scale
// factors out of the sum and is applied once, in the finalize step.
//
// Lookup: each CTA holds a lane-private copy of every codebook in shared memory
// (entry k of lane L at word k*32 + L), so the 32 lanes of a warp always hit 32
// different banks whatever indices they decode. One 32-bit load returns both
// components (C[k][0], C[k][1]); two such loads are re-paired with a byte
// permute into the A registers of rows 2p and 2p+1 (the centroid pairs run
// along output channels, the MMA pairs along K).
//
// Work split: a warp task is (output group of 64 channels, matrix, K chunk).
// Each task writes FP32 partial sums; the last task of an output group to
// arrive (atomic counter, no waiting) sums the partials in a fixed order,
// applies the scales and writes FP16: y (linear) or silu(g)*u (gate/up).
//
// Source of the computation: model card "anemll/anemll-forge-qwen3.8-27B",
// section "Release 0.2: three-bit MLP, token-mixer rotations, distilled
// weights" (2x64 vector LUT, per-channel scales); SiLU as x*sigmoid(x) per
// "ANEMLL ANE LLM conversion pipeline", section "Facts".
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTabWords = 64 * 32;  // one lane-private codebook

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Byte address (relative to the table base) of the lookup for lane index N:
// bits [6N, 6N+6) of the lane's 384-bit string moved to bits [7, 13), OR-ed
// with the lane's own offset (lane*4, plus the matrix's table offset).
template <int N>
__device__ __forceinline__ uint32_t lut_addr(const uint32_t (&w)[12], uint32_t lanebase) {
  constexpr int pos = 6 * N;
  constexpr int wd = pos / 32;
  constexpr int off = pos % 32;
  uint32_t v;
  if constexpr (off >= 7) {
    const uint32_t hi = (wd + 1 < 12) ? w[wd + 1] : 0u;
    v = __funnelshift_r(w[wd], hi, off - 7);
  } else {
    v = w[wd] << (7 - off);
  }
  return (v & 0x1F80u) | lanebase;
}

__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(saddr));
  return v;
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int S, int M, int NT>
__device__ __forceinline__ void mma_step(const uint32_t (&w)[12], uint32_t tab, uint32_t lanebase,
                                         float (&acc)[4][NT][4], const uint32_t (&b)[NT][2]) {
  constexpr int n0 = (S * 4 + M) * 4;
  const uint32_t l0 = lds32(tab + lut_addr<n0 + 0>(w, lanebase));
  const uint32_t l1 = lds32(tab + lut_addr<n0 + 1>(w, lanebase));
  const uint32_t l2 = lds32(tab + lut_addr<n0 + 2>(w, lanebase));
  const uint32_t l3 = lds32(tab + lut_addr<n0 + 3>(w, lanebase));
  uint32_t a[4];
  a[0] = __byte_perm(l0, l1, 0x5410);  // row g   (channel 2p):   inputs k, k+1
  a[1] = __byte_perm(l0, l1, 0x7632);  // row g+8 (channel 2p+1): inputs k, k+1
  a[2] = __byte_perm(l2, l3, 0x5410);  // row g:   inputs k+8, k+9
  a[3] = __byte_perm(l2, l3, 0x7632);  // row g+8: inputs k+8, k+9
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) mma16816(acc[M][nt], a, b[nt]);
}

template <int S, int NT>
__device__ __forceinline__ void kstep(const uint32_t (&w)[12], uint32_t tab, uint32_t lanebase,
                                      float (&acc)[4][NT][4], const uint16_t* __restrict__ xr,
                                      int d_in, int rows, int k0, int g, int t) {
  uint32_t b[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = nt * 8 + g;
    if (r < rows) {
      const uint32_t* xp = reinterpret_cast<const uint32_t*>(xr + (size_t)r * d_in + k0 + S * 16 + 2 * t);
      b[nt][0] = __ldg(xp);
      b[nt][1] = __ldg(xp + 4);
    } else {
      b[nt][0] = 0u;
      b[nt][1] = 0u;
    }
  }
  mma_step<S, 0, NT>(w, tab, lanebase, acc, b);
  mma_step<S, 1, NT>(w, tab, lanebase, acc, b);
  mma_step<S, 2, NT>(w, tab, lanebase, acc, b);
  mma_step<S, 3, NT>(w, tab, lanebase, acc, b);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

template <int NT>
__global__ void __launch_bounds__(kThreads) gemv_kernel(GemvArgs a) {
  __shared__ __align__(16) uint32_t tabs[2 * kTabWords];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  // lane-private codebooks: word k*32 + L of table m holds C_m[k]
  for (int i = tid; i < kTabWords; i += kThreads) tabs[i] = __ldg(a.mats[0].codebook + (i >> 5));
  if (a.n_mats > 1)
    for (int i = tid; i < kTabWords; i += kThreads) tabs[kTabWords + i] = __ldg(a.mats[1].codebook + (i >> 5));
  __syncthreads();

  const int n_groups = a.d_out / kSuChannels;
  const int n_kc = a.d_in / a.kc_len;
  const int per_group = n_kc * a.n_mats;
  const int n_tasks = n_groups * per_group;
  const int task = blockIdx.x * kWarps + warp;
  if (task >= n_tasks) return;

  const int mg = task / per_group;
  const int rem = task % per_group;
  const int mat = rem / n_kc;
  const int kc = rem % n_kc;

  const uint32_t tab = static_cast<uint32_t>(__cvta_generic_to_shared(tabs));
  const uint32_t lanebase = (uint32_t)lane * 4u + (uint32_t)mat * (kTabWords * 4u);

  const int kg_per_chunk = a.kc_len / kSuInputs;
  const int kg_total = a.d_in / kSuInputs;
  const uint4* src = (mat ? a.mats[1].packed : a.mats[0].packed) + ((size_t)mg * kg_total + (size_t)kc * kg_per_chunk) * kSuUint4 + lane;

  float acc[4][NT][4];
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[m][nt][j] = 0.f;

  uint4 nxt[3];
#pragma unroll
  for (int q = 0; q < 3; ++q) nxt[q] = ldg_stream(src + q * 32);

  for (int kg = 0; kg < kg_per_chunk; ++kg) {
    uint32_t w[12];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      w[4 * q + 0] = nxt[q].x;
      w[4 * q + 1] = nxt[q].y;
      w[4 * q + 2] = nxt[q].z;
      w[4 * q + 3] = nxt[q].w;
    }
    if (kg + 1 < kg_per_chunk) {
      const uint4* s2 = src + (size_t)(kg + 1) * kSuUint4;
#pragma unroll
      for (int q = 0; q < 3; ++q) nxt[q] = ldg_stream(s2 + q * 32);
    }
    const int k0 = kc * a.kc_len + kg * kSuInputs;
    kstep<0, NT>(w, tab, lanebase, acc, a.xr, a.d_in, a.rows, k0, g, t);
    kstep<1, NT>(w, tab, lanebase, acc, a.xr, a.d_in, a.rows, k0, g, t);
    kstep<2, NT>(w, tab, lanebase, acc, a.xr, a.d_in, a.rows, k0, g, t);
    kstep<3, NT>(w, tab, lanebase, acc, a.xr, a.d_in, a.rows, k0, g, t);
  }

  // partial sums: accumulator (m, nt) holds rows nt*8+2t (+1) of channels 2p, 2p+1
  float* part = a.partial + ((size_t)kc * a.n_mats + mat) * (size_t)kMaxPassRows * a.d_out;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int p = mg * 32 + m * 8 + g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r0 = nt * 8 + 2 * t;
      if (r0 < a.rows)
        *reinterpret_cast<float2*>(part + (size_t)r0 * a.d_out + 2 * p) = make_float2(acc[m][nt][0], acc[m][nt][2]);
      if (r0 + 1 < a.rows)
        *reinterpret_cast<float2*>(part + (size_t)(r0 + 1) * a.d_out + 2 * p) = make_float2(acc[m][nt][1], acc[m][nt][3]);
    }
  }

  // last arriver of the output group finalizes
  __threadfence();
  __syncwarp();
  unsigned prev = 0;
  if (lane == 0) prev = atomicAdd(a.counters + mg, 1u);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != (unsigned)(per_group - 1)) return;
  __threadfence();

  const int ch = mg * kSuChannels + 2 * lane;  // this lane finalizes channels ch, ch+1
  const size_t mat_stride = (size_t)kMaxPassRows * a.d_out;
  const __half2 s0 = *reinterpret_cast<const __half2*>(a.mats[0].scales + ch);
  const float2 sc0 = __half22float2(s0);
  float2 sc1 = make_float2(0.f, 0.f);
  if (a.mode == kModeSwiglu) sc1 = __half22float2(*reinterpret_cast<const __half2*>(a.mats[1].scales + ch));
  for (int r = 0; r < a.rows; ++r) {
    float2 y0 = make_float2(0.f, 0.f), y1 = make_float2(0.f, 0.f);
    for (int c = 0; c < n_kc; ++c) {
      const float* base = a.partial + (size_t)c * a.n_mats * mat_stride + (size_t)r * a.d_out + ch;
      const float2 v0 = __ldcg(reinterpret_cast<const float2*>(base));
      y0.x += v0.x;
      y0.y += v0.y;
      if (a.mode == kModeSwiglu) {
        const float2 v1 = __ldcg(reinterpret_cast<const float2*>(base + mat_stride));
        y1.x += v1.x;
        y1.y += v1.y;
      }
    }
    float o0, o1;
    if (a.mode == kModeSwiglu) {
      const float g0 = sc0.x * y0.x, g1 = sc0.y * y0.y;
      const float u0 = sc1.x * y1.x, u1 = sc1.y * y1.y;
      o0 = silu_f(g0) * u0;
      o1 = silu_f(g1) * u1;
    } else {
      o0 = sc0.x * y0.x;
      o1 = sc0.y * y0.y;
    }
    *reinterpret_cast<__half2*>(a.out + (size_t)r * a.d_out + ch) = __floats2half2_rn(o0, o1);
  }
  if (lane == 0) a.counters[mg] = 0u;
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st) {
  const int n_tasks = (a.d_out / kSuChannels) * (a.d_in / a.kc_len) * a.n_mats;
  const int grid = (n_tasks + kWarps - 1) / kWarps;
  if (a.rows <= 8)
    gemv_kernel<1><<<grid, kThreads, 0, st>>>(a);
  else if (a.rows <= 16)
    gemv_kernel<2><<<grid, kThreads, 0, st>>>(a);
  else
    gemv_kernel<4><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace vq3
