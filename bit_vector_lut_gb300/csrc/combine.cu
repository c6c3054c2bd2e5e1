// Combine kernels: finish a decode pass from its split-K partial sums.
//
// swiglu_rotate: h = silu(s_g * g) * (s_u * u) for the gate and up pieces, then
// the down projection's online rotation h' = blockdiag(H_b diag(s)) h / sqrt(b),
// written in the fragment order the down decode reads. Sources: model card
// "anemll/anemll-forge-qwen3.8-27B", section "Release 0.2: three-bit MLP,
// token-mixer rotations, distilled weights" (gate/up/down vector LUTs, per-channel
// scales, online Hadamard rotation of each matrix input); SiLU as x*sigmoid(x)
// per "ANEMLL ANE LLM conversion pipeline", section "Facts".
//
// linear_out: y = scale * sum of pieces, FP16.
//
// Pieces of a segment are summed in the order of their CTAs, i.e. in K order,
// so results do not depend on scheduling.
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
namespace {

__device__ __forceinline__ int cta_of(long long x, long long cells, int grid) {
  return (int)(((x + 1) * grid - 1) / cells);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Pieces of one segment: contributing CTAs b0 .. b0+count-1 wrote piece slots
// 0 .. count-1 (the grid never exceeds the number of cells, so every CTA owns at
// least one cell).
struct SegPieces {
  const float* base;  // piece slot 0 of the segment
  int count;
};

__device__ __forceinline__ SegPieces seg_pieces(const PieceMap& pm, int sg) {
  const long long cells = (long long)pm.n_groups * pm.n_kg;
  const long long x0 = (long long)(sg / pm.seg_per_group) * pm.n_kg;
  const int b0 = cta_of(x0, cells, pm.grid), b1 = cta_of(x0 + pm.n_kg - 1, cells, pm.grid);
  SegPieces sp;
  sp.base = pm.pieces + (size_t)sg * pm.max_pieces * 512 * pm.nt;
  sp.count = b1 - b0 + 1;
  return sp;
}

// Sum of item `it` over a segment's pieces, in K order. The loads of a batch
// of up to P pieces are all issued before the first add, so a batch costs one
// round trip to L2.
template <int P>
__device__ __forceinline__ float sum_seg(const SegPieces& sp, int it, int piece_floats) {
  float s = 0.f;
  const float* p = sp.base + it;
  for (int q0 = 0; q0 < sp.count; q0 += P) {
    float v[P];
#pragma unroll
    for (int q = 0; q < P; ++q) v[q] = (q0 + q < sp.count) ? __ldcg(p + (size_t)(q0 + q) * piece_floats) : 0.f;
#pragma unroll
    for (int q = 0; q < P; ++q) s += v[q];
  }
  return s;
}

// Piece item of (row r of the pass, channel c of a 64-channel group).
__device__ __forceinline__ int item_of(int r, int c, int nt_count) {
  const int nt = r >> 3, rr = r & 7, t = rr >> 1, jlo = rr & 1;
  const int pl = c >> 1, m = pl >> 3, g = pl & 7, j = ((c & 1) << 1) | jlo;
  return ((m * nt_count + nt) * 4 + j) * 32 + 4 * g + t;
}

constexpr int kCThreads = 256;

// One CTA: one row of the pass x SPAN channels (a whole number of rotation blocks).
template <int SPAN>
__global__ void __launch_bounds__(kCThreads) swiglu_rotate_kernel(SwigluRotateArgs a) {
  constexpr int G = SPAN / 64;  // 64-channel groups in the span
  __shared__ float hb[SPAN];
  __shared__ SegPieces segs[2 * G];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x;
  const int span0 = blockIdx.x * SPAN;
  const int r = blockIdx.y;  // row within the pass
  const int piece_floats = 512 * a.pm.nt;
  if (tid < 2 * G) segs[tid] = seg_pieces(a.pm, (span0 / 64 + tid / 2) * 2 + (tid & 1));
  __syncthreads();

  const bool live = r < a.rows;
  constexpr int PER = SPAN / kCThreads > 0 ? SPAN / kCThreads : 1;
  constexpr int P = 8;  // pieces per batch
  float gs[PER], us[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) gs[k] = us[k] = 0.f;
  if (live) {
    // one batch: PER channels x 2 matrices x P pieces, all loads in flight together
    int pmax = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int c = tid + k * kCThreads;
      if (c < SPAN) pmax = max(pmax, max(segs[2 * (c >> 6)].count, segs[2 * (c >> 6) + 1].count));
    }
    for (int q0 = 0; q0 < pmax; q0 += P) {
      float vg[PER][P], vu[PER][P];
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int c = tid + k * kCThreads;
        const int q = (c < SPAN) ? (c >> 6) : 0;
        const int it = item_of(r, c & 63, a.pm.nt);
        const SegPieces& sgp = segs[2 * q];
        const SegPieces& sup = segs[2 * q + 1];
#pragma unroll
        for (int j = 0; j < P; ++j) {
          vg[k][j] = (c < SPAN && q0 + j < sgp.count) ? __ldcg(sgp.base + it + (size_t)(q0 + j) * piece_floats) : 0.f;
          vu[k][j] = (c < SPAN && q0 + j < sup.count) ? __ldcg(sup.base + it + (size_t)(q0 + j) * piece_floats) : 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < PER; ++k)
#pragma unroll
        for (int j = 0; j < P; ++j) {
          gs[k] += vg[k][j];
          us[k] += vu[k][j];
        }
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int c = tid + k * kCThreads;
    if (c >= SPAN) continue;
    float hv = 0.f;
    if (live) {
      const int ch = span0 + c;
      const float sg = __half2float(__ushort_as_half(a.scale_gate[ch]));
      const float su = __half2float(__ushort_as_half(a.scale_up[ch]));
      hv = silu_f(sg * gs[k]) * (su * us[k]);
      if (a.signs && ((__ldg(a.signs + (ch >> 5)) >> (ch & 31)) & 1u)) hv = -hv;
    }
    hb[c] = hv;
  }
  __syncthreads();
  // Hadamard butterflies of stride 1 .. block/2 (blocks of `block` channels)
  for (int h = 1; h < a.block && h < SPAN; h <<= 1) {
    for (int q = tid; q < SPAN / 2; q += kCThreads) {
      const int i0 = (q / h) * 2 * h + (q % h), i1 = i0 + h;
      const float x0 = hb[i0], x1 = hb[i1];
      hb[i0] = x0 + x1;
      hb[i1] = x0 - x1;
    }
    __syncthreads();
  }
  const float scale = 1.0f / sqrtf((float)a.block);
  uint16_t* out = reinterpret_cast<uint16_t*>(a.hfrag);
  const int row = a.row0 + r;
  for (int c = tid; c < SPAN; c += kCThreads)
    out[frag_half_index(row, span0 + c, a.n_tiles)] = __half_as_ushort(__float2half_rn(hb[c] * scale));
}

// One CTA: 256 items of one segment's pieces (one thread per item).
__global__ void __launch_bounds__(256) linear_out_kernel(LinearOutArgs a) {
  __shared__ SegPieces seg;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int sg = blockIdx.x;
  const int it = blockIdx.y * 256 + threadIdx.x;  // item of the piece
  if (threadIdx.x == 0) seg = seg_pieces(a.pm, sg);
  __syncthreads();
  const float y = sum_seg<32>(seg, it, 512 * a.pm.nt);
  // item -> (row of the pass, channel): it = ((m*NT + nt)*4 + j)*32 + L
  const int L = it & 31, idx = it >> 5;
  const int j = idx & 3, mnt = idx >> 2, nt = mnt % a.pm.nt, m = mnt / a.pm.nt;
  const int g = L >> 2, t = L & 3;
  const int ch = (sg * 32 + 8 * m + g) * 2 + (j >> 1);
  const int rp = nt * 8 + 2 * t + (j & 1);
  if (rp < a.rows) {
    const float s = __half2float(__ushort_as_half(a.scales[ch]));
    a.out[(size_t)(a.row0 + rp) * a.d_out + ch] = __half_as_ushort(__float2half_rn(s * y));
  }
}

template <typename K, typename A>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t st, const A& args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swiglu_rotate(const SwigluRotateArgs& a, cudaStream_t st) {
  const int span = a.block < 64 ? 64 : a.block;
  const dim3 grid(a.d_inter / span, 8 * a.pm.nt);
  switch (span) {
    case 64: return launch_pdl(swiglu_rotate_kernel<64>, grid, dim3(kCThreads), st, a);
    case 128: return launch_pdl(swiglu_rotate_kernel<128>, grid, dim3(kCThreads), st, a);
    case 256: return launch_pdl(swiglu_rotate_kernel<256>, grid, dim3(kCThreads), st, a);
    case 512: return launch_pdl(swiglu_rotate_kernel<512>, grid, dim3(kCThreads), st, a);
    case 1024: return launch_pdl(swiglu_rotate_kernel<1024>, grid, dim3(kCThreads), st, a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_linear_out(const LinearOutArgs& a, cudaStream_t st) {
  return launch_pdl(linear_out_kernel, dim3(a.d_out / 64, 2 * a.pm.nt), dim3(256), st, a);
}

}  // namespace vq3
