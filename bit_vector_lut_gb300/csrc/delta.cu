// Gated delta-rule token mixer over blocks of 8 tokens.
//
// Source: model card "anemll/anemll-forge-qwen3.8-27B", section "Faster exact
// graph (previous update)", bullet "Gated DeltaNet": tokens are processed in
// 8-row blocks, each needing a triangular solve, done with the exact closed form
// (I + N)^-1 = (I - N)(I + N^2)(I + N^4) for the strictly lower-triangular block.
// The recurrence (a reading of the pages, which name it without writing it out):
//     S_t = alpha_t S_{t-1} + beta_t k_t (v_t - alpha_t S_{t-1}^T k_t)^T,  o_t = S_t^T q_t.
// Over a block of 8 tokens from state S0, with gamma_t = alpha_1 ... alpha_t:
//     N[t][j] = (gamma_t / gamma_j) beta_j (k_t . k_j)        for j < t
//     U      = (I + N)^-1 (V - Gamma K S0)
//     O      = Gamma Q S0 + M U,  M[t][j] = (gamma_t / gamma_j) beta_j (q_t . k_j)  for j <= t
//     S8     = gamma_8 S0 + K^T diag(beta_j gamma_8 / gamma_j) U
// Every column of S, V, U and O is independent of the others, so one CTA takes one
// head and 16 of its d_v columns, keeps that slice of the state in shared memory
// and walks the blocks in order. FP32 arithmetic, FP16 inputs and outputs.
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
namespace {

constexpr int kB = 8;       // tokens per block
constexpr int kCols = 16;   // d_v columns per CTA
constexpr int kDThreads = 128;

__device__ __forceinline__ float h2f(uint16_t v) { return __half2float(__ushort_as_half(v)); }

__global__ void __launch_bounds__(kDThreads) delta_rule_kernel(const uint16_t* __restrict__ q,
                                                                 const uint16_t* __restrict__ k,
                                                                 const uint16_t* __restrict__ v,
                                                                 const float* __restrict__ beta,
                                                                 const float* __restrict__ alpha, int tokens, int heads,
                                                                 int d_k, int d_v, float* __restrict__ state,
                                                                 uint16_t* __restrict__ out) {
  extern __shared__ float sm[];
  float* Ss = sm;                    // [d_k][16] state slice
  float* Ks = Ss + d_k * kCols;      // [8][d_k]
  float* Qs = Ks + kB * d_k;         // [8][d_k]
  __shared__ float Vs[kB][kCols], KS[kB][kCols], QS[kB][kCols], R[kB][kCols], U[kB][kCols];
  __shared__ float KK[kB][kB], QK[kB][kB], P[kB][kB], T1[kB][kB], T2[kB][kB];
  __shared__ float be[kB], ga[kB];
  const int tid = threadIdx.x;
  const int h = blockIdx.x, c0 = blockIdx.y * kCols;
  float* Sg = state + (size_t)h * d_k * d_v;
  for (int e = tid; e < d_k * kCols; e += kDThreads) Ss[e] = Sg[(size_t)(e / kCols) * d_v + c0 + e % kCols];
  const int t_ = tid / kCols, c_ = tid % kCols;  // (token, column) of this thread in the 8 x 16 phases

  for (int b0 = 0; b0 < tokens; b0 += kB) {
    // ---- block inputs; tokens past the last act as k = q = v = 0, beta = 0, alpha = 1
    for (int e = tid; e < kB * d_k; e += kDThreads) {
      const int t = e / d_k, i = e % d_k;
      const bool ok = b0 + t < tokens;
      const size_t o = ((size_t)(b0 + t) * heads + h) * d_k + i;
      Ks[e] = ok ? h2f(k[o]) : 0.f;
      Qs[e] = ok ? h2f(q[o]) : 0.f;
    }
    {
      const bool ok = b0 + t_ < tokens;
      Vs[t_][c_] = ok ? h2f(v[((size_t)(b0 + t_) * heads + h) * d_v + c0 + c_]) : 0.f;
    }
    if (tid < kB) {
      const bool ok = b0 + tid < tokens;
      be[tid] = ok ? beta[(size_t)(b0 + tid) * heads + h] : 0.f;
      ga[tid] = ok ? alpha[(size_t)(b0 + tid) * heads + h] : 1.f;
    }
    __syncthreads();
    if (tid == 0)
      for (int t = 1; t < kB; ++t) ga[t] *= ga[t - 1];  // gamma_t = alpha_1 ... alpha_t
    // ---- k_t . k_j, q_t . k_j (thread < 64: KK, else QK), and K S0, Q S0 for the slice
    {
      const int pr = tid & 63, t = pr / kB, j = pr % kB;
      const float* a = (tid < 64 ? Ks : Qs) + t * d_k;
      const float* bb = Ks + j * d_k;
      float s = 0.f;
      for (int i = 0; i < d_k; ++i) s = fmaf(a[i], bb[i], s);
      if (tid < 64)
        KK[t][j] = s;
      else
        QK[t][j] = s;
      float ks = 0.f, qs = 0.f;
      for (int i = 0; i < d_k; ++i) {
        const float sv = Ss[i * kCols + c_];
        ks = fmaf(Ks[t_ * d_k + i], sv, ks);
        qs = fmaf(Qs[t_ * d_k + i], sv, qs);
      }
      KS[t_][c_] = ks;
      QS[t_][c_] = qs;
    }
    __syncthreads();
    // ---- N (strictly lower) and the closed-form inverse P = (I - N)(I + N^2)(I + N^4)
    if (tid < 64) {
      const int t = tid / kB, j = tid % kB;
      P[t][j] = j < t ? ga[t] / ga[j] * be[j] * KK[t][j] : 0.f;  // P holds N for now
    }
    R[t_][c_] = Vs[t_][c_] - ga[t_] * KS[t_][c_];
    __syncthreads();
    if (tid < 64) {  // T1 = N^2
      const int t = tid / kB, j = tid % kB;
      float s = 0.f;
      for (int m = 0; m < kB; ++m) s = fmaf(P[t][m], P[m][j], s);
      T1[t][j] = s;
    }
    __syncthreads();
    if (tid < 64) {  // T2 = N^4
      const int t = tid / kB, j = tid % kB;
      float s = 0.f;
      for (int m = 0; m < kB; ++m) s = fmaf(T1[t][m], T1[m][j], s);
      T2[t][j] = s;
    }
    __syncthreads();
    if (tid < 64) {  // KK <- (I - N)(I + N^2)
      const int t = tid / kB, j = tid % kB;
      float s = 0.f;
      for (int m = 0; m < kB; ++m) {
        const float a = (t == m ? 1.f : 0.f) - P[t][m];
        const float bb = (m == j ? 1.f : 0.f) + T1[m][j];
        s = fmaf(a, bb, s);
      }
      KK[t][j] = s;
    }
    __syncthreads();
    if (tid < 64) {  // P <- KK (I + N^4)
      const int t = tid / kB, j = tid % kB;
      float s = 0.f;
      for (int m = 0; m < kB; ++m) s = fmaf(KK[t][m], (m == j ? 1.f : 0.f) + T2[m][j], s);
      P[t][j] = s;
    }
    __syncthreads();
    // ---- U = P R
    {
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < kB; ++j) s = fmaf(P[t_][j], R[j][c_], s);
      U[t_][c_] = s;
    }
    __syncthreads();
    // ---- O = Gamma Q S0 + M U
    {
      float s = ga[t_] * QS[t_][c_];
      for (int j = 0; j <= t_; ++j) s = fmaf(ga[t_] / ga[j] * be[j] * QK[t_][j], U[j][c_], s);
      if (b0 + t_ < tokens)
        out[((size_t)(b0 + t_) * heads + h) * d_v + c0 + c_] = __half_as_ushort(__float2half_rn(s));
    }
    // ---- S = gamma_8 S0 + K^T diag(beta_j gamma_8 / gamma_j) U
    for (int i = tid; i < d_k; i += kDThreads) {
      float w[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) w[j] = Ks[j * d_k + i] * (be[j] * ga[kB - 1] / ga[j]);
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        float s = ga[kB - 1] * Ss[i * kCols + c];
#pragma unroll
        for (int j = 0; j < kB; ++j) s = fmaf(w[j], U[j][c], s);
        Ss[i * kCols + c] = s;
      }
    }
    __syncthreads();
  }
  for (int e = tid; e < d_k * kCols; e += kDThreads) Sg[(size_t)(e / kCols) * d_v + c0 + e % kCols] = Ss[e];
}

}  // namespace

cudaError_t launch_delta_rule(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* beta,
                              const float* alpha, int tokens, int heads, int d_k, int d_v, float* state,
                              uint16_t* out, cudaStream_t st) {
  const size_t smem = (size_t)(d_k * kCols + 2 * kB * d_k) * sizeof(float);
  const dim3 grid((unsigned)heads, (unsigned)(d_v / kCols));
  delta_rule_kernel<<<grid, kDThreads, smem, st>>>(q, k, v, beta, alpha, tokens, heads, d_k, d_v, state, out);
  return cudaGetLastError();
}

}  // namespace vq3
