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
// Every column of S, V, U and O is independent of the others, so a CTA takes one
// head and 16 of its d_v columns and walks the blocks in order. Two kernels: the
// tensor-core one below (d_k a multiple of 16 up to 128) and, for other d_k, one in
// FP32 on CUDA cores that keeps the state slice in shared memory.
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
VQ3_BOUNDS_RECORD(delta)
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
  const size_t n_state = (size_t)heads * d_k * d_v, n_qk = (size_t)tokens * heads * d_k, n_v = (size_t)tokens * heads * d_v;
  for (int e = tid; e < d_k * kCols; e += kDThreads)
    Ss[e] = VQ3_IN((size_t)h * d_k * d_v + (size_t)(e / kCols) * d_v + c0 + e % kCols, n_state, 1)
                ? Sg[(size_t)(e / kCols) * d_v + c0 + e % kCols] : 0.f;
  const int t_ = tid / kCols, c_ = tid % kCols;  // (token, column) of this thread in the 8 x 16 phases

  for (int b0 = 0; b0 < tokens; b0 += kB) {
    // ---- block inputs; tokens past the last act as k = q = v = 0, beta = 0, alpha = 1
    for (int e = tid; e < kB * d_k; e += kDThreads) {
      const int t = e / d_k, i = e % d_k;
      const size_t o = ((size_t)(b0 + t) * heads + h) * d_k + i;
      const bool ok = b0 + t < tokens && VQ3_IN(o, n_qk, 2);
      Ks[e] = ok ? h2f(k[o]) : 0.f;
      Qs[e] = ok ? h2f(q[o]) : 0.f;
    }
    {
      const bool ok = b0 + t_ < tokens && VQ3_IN(((size_t)(b0 + t_) * heads + h) * d_v + c0 + c_, n_v, 3);
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
      if (b0 + t_ < tokens && VQ3_IN(((size_t)(b0 + t_) * heads + h) * d_v + c0 + c_, n_v, 4))
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
  for (int e = tid; e < d_k * kCols; e += kDThreads)
    if (VQ3_IN((size_t)h * d_k * d_v + (size_t)(e / kCols) * d_v + c0 + e % kCols, n_state, 5))
      Sg[(size_t)(e / kCols) * d_v + c0 + e % kCols] = Ss[e];
}


// ---------------------------------------------------------------- tensor-core path (d_k = 16 KS <= 128)
//
// One CTA of KS warps per (head, 16 columns of d_v). The state slice is held transposed,
// S^T [16 columns][d_k], as the accumulators of m16n8k16 tiles (n-tile n: d_k 8n .. 8n+7),
// warp w holding n-tiles 2w and 2w+1 (d_k 16w .. 16w+15): that is also the A-operand layout of
// k-step w of the next product S^T [K; Q]^T, so the state never leaves the registers between
// blocks. The FP32 operands that enter the tensor cores (the state, the weighted U) are split
// into two FP16 parts, hi = fp16(x) and lo = fp16(x - hi), and multiplied as two MMAs into FP32
// accumulators (about 22 bits of each operand; K and Q are FP16 inputs).
// Per chunk of up to 64 tokens: K, Q, V, alpha, beta staged in shared memory; the state-
// independent parts of the 8-token blocks first, warp w taking blocks w, w + KS, ... (K K^T and
// Q K^T as one 16 x 8 tile, then N, the closed-form P = (I - N)(I + N^2)(I + N^4), M and the
// weights); then the blocks in order:
//     [X_K | X_Q] = S^T [K; Q]^T   (each warp its k-step; the partials added in warp order)
//     R^T = V^T - X_K Gamma,  U^T = R^T P^T,  O^T = X_Q Gamma + U^T M^T   (every warp, redundantly)
//     S^T = gamma_8 S^T + (U diag(w))^T K,  w_j = beta_j gamma_8 / gamma_j   (each warp its tiles)

constexpr int kTcChunk = 64;  // tokens staged at a time (8 blocks)
constexpr int kTcBlocks = kTcChunk / 8;

__device__ __forceinline__ void mma_tc(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (x, y) -> FP16 pair hi and the pair of what hi leaves, lo.
__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x, y);
  const float2 e = __half22float2(h);
  const __half2 l = __floats2half2_rn(x - e.x, y - e.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Dynamic shared memory of the kernel (bytes from the base; every part 16-byte aligned).
template <int KS>
struct TcSmem {
  static constexpr int DK = 16 * KS;
  static constexpr int RS = DK + 8;  // staged row stride in halves: 4 words past a multiple of 32
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kQ = kK + kTcChunk * RS * 2;
  static constexpr uint32_t kV = kQ + kTcChunk * RS * 2;       // FP16 [64][16]
  static constexpr uint32_t kAl = kV + kTcChunk * 16 * 2;      // alpha [64], beta [64]
  static constexpr uint32_t kP = kAl + 2 * kTcChunk * 4;       // P, M [blocks][8][8]
  static constexpr uint32_t kG = kP + 2 * kTcBlocks * 64 * 4;  // gamma, w [blocks][8]
  // phase-1 scratch [KS][6][8][8] and, later in the chunk, the X partials [2][KS][2][32][4]
  static constexpr uint32_t kU = kG + 2 * kTcBlocks * 8 * 4;
  static constexpr uint32_t kUBytes = (uint32_t)KS * 2048u;
  static constexpr uint32_t kTotal = kU + kUBytes;
};

// z = (dx I + x)(dy I + y) for 8 x 8 matrices in a warp's shared scratch, two entries per lane.
__device__ __forceinline__ void mul8(float (*x)[8], float (*y)[8], float (*z)[8], float dx, float dy, int lane) {
  float r2[2];
#pragma unroll
  for (int e2 = 0; e2 < 2; ++e2) {
    const int e = lane + 32 * e2, ti = e >> 3, j = e & 7;
    float s = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) s = fmaf((ti == m ? dx : 0.f) + x[ti][m], (m == j ? dy : 0.f) + y[m][j], s);
    r2[e2] = s;
  }
  __syncwarp();
  z[lane >> 3][lane & 7] = r2[0];
  z[(lane + 32) >> 3][lane & 7] = r2[1];
  __syncwarp();
}

template <int KS>
__global__ void __launch_bounds__(32 * KS, 1) delta_rule_tc_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                                                                const uint16_t* __restrict__ v,
                                                                const float* __restrict__ beta,
                                                                const float* __restrict__ alpha, int tokens, int heads,
                                                                int d_v, float* __restrict__ state,
                                                                uint16_t* __restrict__ out) {
  using L = TcSmem<KS>;
  constexpr int DK = L::DK, RS = L::RS, NT = 32 * KS;
  extern __shared__ __align__(16) unsigned char dsm[];
  uint16_t* Ks = reinterpret_cast<uint16_t*>(dsm + L::kK);
  uint16_t* Qs = reinterpret_cast<uint16_t*>(dsm + L::kQ);
  uint16_t (*Vh)[16] = reinterpret_cast<uint16_t (*)[16]>(dsm + L::kV);
  float* Al = reinterpret_cast<float*>(dsm + L::kAl);
  float* Be = Al + kTcChunk;
  float (*Pm)[8][8] = reinterpret_cast<float (*)[8][8]>(dsm + L::kP);
  float (*Mm)[8][8] = Pm + kTcBlocks;
  float (*Gm)[8] = reinterpret_cast<float (*)[8]>(dsm + L::kG);
  float (*Wm)[8] = Gm + kTcBlocks;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  float (*Sc)[8][8] = reinterpret_cast<float (*)[8][8]>(dsm + L::kU + (uint32_t)warp * 1536u);  // 6 of them
  float* Xp = reinterpret_cast<float*>(dsm + L::kU);  // [2][KS][2][32][4]
  const int h = blockIdx.x, c0 = blockIdx.y * 16;
  float* Sg = state + (size_t)h * DK * d_v + c0;
  const size_t n_state = (size_t)heads * DK * d_v, n_qk = (size_t)tokens * heads * DK, n_v = (size_t)tokens * heads * d_v;

  // this warp's tiles of the state slice: acc[n] = S^T[g, g+8][16 warp + 8n + 2t, +1]
  float acc[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const int d = 16 * warp + 8 * n + 2 * t;
    if (!VQ3_IN((size_t)h * DK * d_v + c0 + (size_t)(d + 1) * d_v + g + 8, n_state, 11)) {
      acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
      continue;
    }
    acc[n][0] = Sg[(size_t)d * d_v + g];
    acc[n][1] = Sg[(size_t)(d + 1) * d_v + g];
    acc[n][2] = Sg[(size_t)d * d_v + g + 8];
    acc[n][3] = Sg[(size_t)(d + 1) * d_v + g + 8];
  }

  for (int base = 0; base < tokens; base += kTcChunk) {
    const int nt = tokens - base < kTcChunk ? tokens - base : kTcChunk;
    const int nb = (nt + 7) / 8;
    // ---- stage K, Q, V (16-byte copies), alpha, beta; tokens past the last are zero (beta 0, alpha 1)
    const uint32_t ks = static_cast<uint32_t>(__cvta_generic_to_shared(Ks));
    const uint32_t qs = static_cast<uint32_t>(__cvta_generic_to_shared(Qs));
    for (int i = tid; i < nb * 8 * (DK / 8); i += NT) {
      const int tk = i / (DK / 8), c = i % (DK / 8);
      const uint32_t off = (uint32_t)(tk * RS + c * 8) * 2u;
      if (tk < nt && VQ3_IN(((size_t)(base + tk) * heads + h) * DK + c * 8 + 7, n_qk, 12)) {
        const size_t src = ((size_t)(base + tk) * heads + h) * DK + c * 8;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ks + off), "l"(k + src) : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(qs + off), "l"(q + src) : "memory");
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(ks + off), "r"(0u) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(qs + off), "r"(0u) : "memory");
      }
    }
    for (int i = tid; i < nb * 8 * 2; i += NT) {  // two 16-byte halves of each token's 16 columns
      const int tk = i >> 1, c = (i & 1) * 8;
      const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(&Vh[tk][c]));
      if (tk < nt && VQ3_IN(((size_t)(base + tk) * heads + h) * d_v + c0 + c + 7, n_v, 13))
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                     "l"(v + ((size_t)(base + tk) * heads + h) * d_v + c0 + c) : "memory");
      else
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int i = tid; i < nb * 8; i += NT) {
      Al[i] = i < nt ? alpha[(size_t)(base + i) * heads + h] : 1.f;
      Be[i] = i < nt ? beta[(size_t)(base + i) * heads + h] : 0.f;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();  // every thread's copies and stores are visible

    // ---- the state-independent parts of every block: warp w takes blocks w, w + KS, ...
    for (int b = warp; b < nb; b += KS) {
      const int tb = 8 * b;
      float (*Nn)[8] = Sc[0], (*N2)[8] = Sc[1], (*N4)[8] = Sc[2], (*Am)[8] = Sc[3], (*KK)[8] = Sc[4], (*QK)[8] = Sc[5];
      float gk[4] = {0.f, 0.f, 0.f, 0.f};  // rows g: k_g . k_{2t}, k_g . k_{2t+1}; rows g+8: q_g . k_..
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const uint16_t* kr = Ks + (tb + g) * RS + 16 * s + 2 * t;
        const uint16_t* qr = Qs + (tb + g) * RS + 16 * s + 2 * t;
        const uint32_t k0 = *reinterpret_cast<const uint32_t*>(kr), k1 = *reinterpret_cast<const uint32_t*>(kr + 8);
        const uint32_t q0 = *reinterpret_cast<const uint32_t*>(qr), q1 = *reinterpret_cast<const uint32_t*>(qr + 8);
        const uint32_t a[4] = {k0, q0, k1, q1};
        mma_tc(gk, a, k0, k1);
      }
      KK[g][2 * t] = gk[0];
      KK[g][2 * t + 1] = gk[1];
      QK[g][2 * t] = gk[2];
      QK[g][2 * t + 1] = gk[3];
      if (lane == 0) {
        float gam = 1.f;
        for (int j = 0; j < 8; ++j) {  // gamma_j = alpha_1 ... alpha_j; beta, then the weights below
          gam *= Al[tb + j];
          Gm[b][j] = gam;
          Wm[b][j] = Be[tb + j];
        }
      }
      __syncwarp();
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {  // N (strictly lower) and M (lower with the diagonal)
        const int e = lane + 32 * e2, ti = e >> 3, j = e & 7;
        const float f = Gm[b][ti] / Gm[b][j] * Wm[b][j];
        Nn[ti][j] = j < ti ? f * KK[ti][j] : 0.f;
        Mm[b][ti][j] = j <= ti ? f * QK[ti][j] : 0.f;
      }
      __syncwarp();
      mul8(Nn, Nn, N2, 0.f, 0.f, lane);  // N^2
      mul8(N2, N2, N4, 0.f, 0.f, lane);  // N^4
      Nn[lane >> 3][lane & 7] = -Nn[lane >> 3][lane & 7];  // then (I - N)(I + N^2)
      Nn[(lane + 32) >> 3][lane & 7] = -Nn[(lane + 32) >> 3][lane & 7];
      __syncwarp();
      mul8(Nn, N2, Am, 1.f, 1.f, lane);
      mul8(Am, N4, Pm[b], 0.f, 1.f, lane);  // P = A (I + N^4)
      if (lane < 8) Wm[b][lane] = Wm[b][lane] * Gm[b][7] / Gm[b][lane];  // w_j = beta_j gamma_8 / gamma_j
      __syncwarp();
    }
    __syncthreads();  // every block's P, M, gamma and w are visible; the scratch is free for X

    // ---- the blocks in order
    for (int b = 0; b < nb; ++b) {
      const int tb = 8 * b;
      // this warp's k-step of [X_K | X_Q] = S^T [K; Q]^T (d_k 16 warp .. + 15)
      {
        uint32_t ah[4], al[4];
        split2(acc[0][0], acc[0][1], ah[0], al[0]);
        split2(acc[0][2], acc[0][3], ah[1], al[1]);
        split2(acc[1][0], acc[1][1], ah[2], al[2]);
        split2(acc[1][2], acc[1][3], ah[3], al[3]);
        const uint16_t* kr = Ks + (tb + g) * RS + 16 * warp + 2 * t;
        const uint16_t* qr = Qs + (tb + g) * RS + 16 * warp + 2 * t;
        const uint32_t k0 = *reinterpret_cast<const uint32_t*>(kr), k1 = *reinterpret_cast<const uint32_t*>(kr + 8);
        const uint32_t q0 = *reinterpret_cast<const uint32_t*>(qr), q1 = *reinterpret_cast<const uint32_t*>(qr + 8);
        float xk[4] = {0.f, 0.f, 0.f, 0.f}, xq[4] = {0.f, 0.f, 0.f, 0.f};
        mma_tc(xk, ah, k0, k1);
        mma_tc(xq, ah, q0, q1);
        mma_tc(xk, al, k0, k1);
        mma_tc(xq, al, q0, q1);
        // [parity][warp][K | Q][lane][4]: 16-byte stores, lanes 16 bytes apart (double-buffered by parity)
        float4* xp = reinterpret_cast<float4*>(Xp) + ((b & 1) * KS + warp) * 64 + lane;
        xp[0] = make_float4(xk[0], xk[1], xk[2], xk[3]);
        xp[32] = make_float4(xq[0], xq[1], xq[2], xq[3]);
      }
      __syncthreads();  // every warp's partial is in shared memory
      // the partials added in warp (= k-step) order: (K S)^T and (Q S)^T at [g][2t], [g][2t+1],
      // [g+8][2t], [g+8][2t+1] (every warp forms the same sums)
      float xk[4] = {0.f, 0.f, 0.f, 0.f}, xq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w2 = 0; w2 < KS; ++w2) {
        const float4* xp = reinterpret_cast<const float4*>(Xp) + ((b & 1) * KS + w2) * 64 + lane;
        const float4 pk = xp[0], pq = xp[32];
        xk[0] += pk.x;
        xk[1] += pk.y;
        xk[2] += pk.z;
        xk[3] += pk.w;
        xq[0] += pq.x;
        xq[1] += pq.y;
        xq[2] += pq.z;
        xq[3] += pq.w;
      }
      const float* gm = Gm[b];
      const int j0 = 2 * t, j1 = 2 * t + 1;
      const float r0 = h2f(Vh[tb + j0][g]) - gm[j0] * xk[0], r1 = h2f(Vh[tb + j1][g]) - gm[j1] * xk[1];
      const float r2 = h2f(Vh[tb + j0][g + 8]) - gm[j0] * xk[2], r3 = h2f(Vh[tb + j1][g + 8]) - gm[j1] * xk[3];
      // U^T[c][i] = sum_j P[i][j] R^T[c][j]: this lane's two j, then the four lanes of row g
      float ulo[8], uhi[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 pp = *reinterpret_cast<const float2*>(&Pm[b][i][j0]);  // P[i][2t], P[i][2t+1]
        ulo[i] = fmaf(pp.y, r1, pp.x * r0);
        uhi[i] = fmaf(pp.y, r3, pp.x * r2);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ulo[i] += __shfl_xor_sync(0xffffffffu, ulo[i], 1);
        uhi[i] += __shfl_xor_sync(0xffffffffu, uhi[i], 1);
        ulo[i] += __shfl_xor_sync(0xffffffffu, ulo[i], 2);
        uhi[i] += __shfl_xor_sync(0xffffffffu, uhi[i], 2);
      }
      // this lane's entries (selected, not indexed: the arrays stay in registers)
      float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        u0 = i == j0 ? ulo[i] : u0;
        u1 = i == j1 ? ulo[i] : u1;
        u2 = i == j0 ? uhi[i] : u2;
        u3 = i == j1 ? uhi[i] : u3;
      }
      if (warp == 0) {
        // O^T[c][i] = gamma_i X_Q[c][i] + sum_{j <= i} M[i][j] U^T[c][j] (the full sum over j: M is zero above)
        float olo[8], ohi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 mm = *reinterpret_cast<const float2*>(&Mm[b][i][j0]);  // M[i][2t], M[i][2t+1]
          olo[i] = fmaf(mm.y, u1, mm.x * u0);
          ohi[i] = fmaf(mm.y, u3, mm.x * u2);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          olo[i] += __shfl_xor_sync(0xffffffffu, olo[i], 1);
          ohi[i] += __shfl_xor_sync(0xffffffffu, ohi[i], 1);
          olo[i] += __shfl_xor_sync(0xffffffffu, olo[i], 2);
          ohi[i] += __shfl_xor_sync(0xffffffffu, ohi[i], 2);
        }
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          s0 = i == j0 ? olo[i] : s0;
          s1 = i == j1 ? olo[i] : s1;
          s2 = i == j0 ? ohi[i] : s2;
          s3 = i == j1 ? ohi[i] : s3;
        }
        const float o0 = fmaf(gm[j0], xq[0], s0), o1 = fmaf(gm[j1], xq[1], s1);
        const float o2 = fmaf(gm[j0], xq[2], s2), o3 = fmaf(gm[j1], xq[3], s3);
        const int tk0 = base + tb + j0, tk1 = base + tb + j1;
        if (tk0 < tokens && VQ3_IN(((size_t)tk0 * heads + h) * d_v + c0 + g + 8, n_v, 14)) {
          uint16_t* o = out + ((size_t)tk0 * heads + h) * d_v + c0;
          o[g] = __half_as_ushort(__float2half_rn(o0));
          o[g + 8] = __half_as_ushort(__float2half_rn(o2));
        }
        if (tk1 < tokens && VQ3_IN(((size_t)tk1 * heads + h) * d_v + c0 + g + 8, n_v, 14)) {
          uint16_t* o = out + ((size_t)tk1 * heads + h) * d_v + c0;
          o[g] = __half_as_ushort(__float2half_rn(o1));
          o[g + 8] = __half_as_ushort(__float2half_rn(o3));
        }
      }
      // this warp's state tiles: S^T <- gamma_8 S^T + W^T K with W^T[c][j] = U^T[c][j] w_j (tokens
      // 8 .. 15 of the k-step are zero)
      uint32_t wh[4], wl[4];
      split2(u0 * Wm[b][j0], u1 * Wm[b][j1], wh[0], wl[0]);
      split2(u2 * Wm[b][j0], u3 * Wm[b][j1], wh[1], wl[1]);
      wh[2] = wh[3] = wl[2] = wl[3] = 0u;
      const float g8 = gm[7];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int d = 16 * warp + 8 * n + g;
        const uint16_t kv0 = Ks[(tb + j0) * RS + d], kv1 = Ks[(tb + j1) * RS + d];
        const uint32_t bk = (uint32_t)kv0 | ((uint32_t)kv1 << 16);
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[n][r] *= g8;
        mma_tc(acc[n], wh, bk, 0u);
        mma_tc(acc[n], wl, bk, 0u);
      }
    }
    __syncthreads();  // the staged chunk and the partials are read no more
  }
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const int d = 16 * warp + 8 * n + 2 * t;
    if (!VQ3_IN((size_t)h * DK * d_v + c0 + (size_t)(d + 1) * d_v + g + 8, n_state, 15)) continue;
    Sg[(size_t)d * d_v + g] = acc[n][0];
    Sg[(size_t)(d + 1) * d_v + g] = acc[n][1];
    Sg[(size_t)d * d_v + g + 8] = acc[n][2];
    Sg[(size_t)(d + 1) * d_v + g + 8] = acc[n][3];
  }
}

template <int KS>
cudaError_t launch_delta_tc(dim3 grid, const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* beta,
                            const float* alpha, int tokens, int heads, int d_v, float* state, uint16_t* out,
                            cudaStream_t st) {
  constexpr int smem = (int)TcSmem<KS>::kTotal;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(delta_rule_tc_kernel<KS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  delta_rule_tc_kernel<KS><<<grid, 32 * KS, smem, st>>>(q, k, v, beta, alpha, tokens, heads, d_v, state, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_delta_rule(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* beta,
                              const float* alpha, int tokens, int heads, int d_k, int d_v, float* state,
                              uint16_t* out, cudaStream_t st) {
  const dim3 grid((unsigned)heads, (unsigned)(d_v / kCols));
  const bool al = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16 == 0;
  if (d_k % 16 == 0 && d_k <= 128 && al) {  // the tensor-core path (16-byte staging of q, k and v)
    switch (d_k / 16) {
      case 1: return launch_delta_tc<1>(grid, q, k, v, beta, alpha, tokens, heads, d_v, state, out, st);
      case 2: return launch_delta_tc<2>(grid, q, k, v, beta, alpha, tokens, heads, d_v, state, out, st);
      case 3: return launch_delta_tc<3>(grid, q, k, v, beta, alpha, tokens, heads, d_v, state, out, st);
      case 4: return launch_delta_tc<4>(grid, q, k, v, beta, alpha, tokens, heads, d_v, state, out, st);
      case 5: return launch_delta_tc<5>(grid, q, k, v, beta, alpha, tokens, heads, d_v, state, out, st);
      case 6: return launch_delta_tc<6>(grid, q, k, v, beta, alpha, tokens, heads, d_v, state, out, st);
      case 7: return launch_delta_tc<7>(grid, q, k, v, beta, alpha, tokens, heads, d_v, state, out, st);
      default: return launch_delta_tc<8>(grid, q, k, v, beta, alpha, tokens, heads, d_v, state, out, st);
    }
  }
  const size_t smem = (size_t)(d_k * kCols + 2 * kB * d_k) * sizeof(float);
  delta_rule_kernel<<<grid, kDThreads, smem, st>>>(q, k, v, beta, alpha, tokens, heads, d_k, d_v, state, out);
  return cudaGetLastError();
}

}  // namespace vq3
