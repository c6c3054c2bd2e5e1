// VQ3 GEMM for small row counts (T <= 32 per pass): weight streaming on the
// m16n8k16 tensor-core path with FP32 accumulation.
//
// What it computes (model card "anemll/anemll-forge-qwen3.8-27B", section
// "Release 0.2: three-bit MLP, token-mixer rotations, distilled weights": a
// 2x64 vector LUT per matrix, one six-bit index per output pair and input,
// per-channel scales; SiLU per "ANEMLL ANE LLM conversion pipeline", "Facts"):
//   y[r][2p+c] = scale[2p+c] * sum_i C[idx[p][i]][c] * x'[r][i]
// and, for gate/up, h = silu(y_gate) * y_up.
//
// Why m16n8k16 and not tcgen05 here: a tcgen05.mma instruction takes the same
// time for any N up to 256, so at N = 8..32 it would absorb ~5 indices per clock
// per SM, a sixth of what streaming the indices at HBM speed needs; the m16n8
// path absorbs ~60, which leaves the decode (shift, mask, shared-memory lookup,
// byte permute per index) as the limit.
//
// Lookup: each CTA holds a lane-private copy of every codebook in shared memory
// (entry k of lane L at word k*32 + L), so the 32 lanes of a warp always hit 32
// different banks whatever indices they decode. One 32-bit load returns both
// components (C[k][0], C[k][1]); two such loads are re-paired with a byte
// permute into the A registers of rows 2p and 2p+1 (the centroid pairs run
// along output channels, the MMA pairs along K).
//
// Work split: the (output group of 64 channels x matrix) "segments" times the
// 64-input column groups form cells; every CTA of a persistent grid owns a
// contiguous run of cells, and its eight warps take the run's cells in turn.
// Each warp keeps two or three cells of index strings and activation
// fragments in flight in shared memory (cp.async). At the end of each segment the warps' accumulators are
// summed in shared memory and written as one partial sum ("piece"). The
// combine kernels (combine.cu) sum a segment's pieces in K order
// (deterministic) and apply the scales, SwiGLU and the next rotation.
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
namespace {

constexpr int kThreads = kDecWarps * 32;
constexpr int kTabWords = 64 * 32;

// Not volatile: a pure function of its registers, so the compiler may schedule
// the lookups of later steps ahead of it.
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared-memory address of the lookup for lane index N: bits [6N, 6N+6) of the
// lane's 384-bit string moved to bits [7, 13) (entry stride 32 lanes x 4 bytes),
// OR-ed with the lane's own column and the matrix's table offset.
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

// The lookup tables are placed at a 16 KB-aligned shared address (inside the
// dynamic shared memory, which is over-allocated by 16 KB for that), so the table
// base, the lane's column and the matrix's table offset are disjoint bit fields
// of one 32-bit shared address and a lookup needs no add: shift, LOP3, load.
constexpr uint32_t kTabAlign = 16384;

// The tables are read-only while the cells are decoded, so the load is a pure
// function of its address (not volatile, no memory clobber): free to reorder.
__device__ __forceinline__ uint32_t lut(uint32_t saddr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(saddr));
  return v;
}

// Prefetch: every lane copies its own operands of a cell (its 48-byte index
// string and the 32*NT bytes of B fragments) into its warp's slot of a shared-
// memory ring with cp.async, kSlots cells ahead, and later reads back exactly
// the bytes it copied, so no other lane is involved.
struct Ring {
  static constexpr int kSlots = 3;
  static constexpr int kSlotBytes = 1536;  // one lane-fragment index string set (a super-unit)
  static constexpr int kWarpBytes = kSlots * kSlotBytes;
};

// Column groups of activation fragments staged per chunk (NT KB each).
template <int NT>
struct Xs {
  static constexpr int kKg = NT == 1 ? 32 : (NT == 2 ? 16 : 8);
  static constexpr int kBytes = kKg * NT * 1024;
  // per-segment reduction buffer when warps split K (at most kDecWarps / 2 segments)
  static constexpr int kRedBytes = (kDecWarps / 2) * 512 * NT * 4;
};

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr) : "memory");
  return v;
}

// slot layout (per warp): [q=0..2][32 lanes][16 B] index words
__device__ __forceinline__ void copy_su(uint32_t slot, int lane, const uint4* su_lane) {
#pragma unroll
  for (int q = 0; q < 3; ++q) cp_async16(slot + (uint32_t)(q * 512 + lane * 16), su_lane + q * 32);
}

template <int S, int M, int NT>
__device__ __forceinline__ void mma_step(const uint32_t (&w)[12], uint32_t lanebase, float (&acc)[4][NT][4],
                                         const uint32_t (&b)[NT][8]) {
  constexpr int n0 = (S * 4 + M) * 4;
  const uint32_t l0 = lut(lut_addr<n0 + 0>(w, lanebase));
  const uint32_t l1 = lut(lut_addr<n0 + 1>(w, lanebase));
  const uint32_t l2 = lut(lut_addr<n0 + 2>(w, lanebase));
  const uint32_t l3 = lut(lut_addr<n0 + 3>(w, lanebase));
  uint32_t a[4];
  a[0] = __byte_perm(l0, l1, 0x5410);  // row g   (channel 2p):   inputs k, k+1
  a[1] = __byte_perm(l0, l1, 0x7632);  // row g+8 (channel 2p+1): inputs k, k+1
  a[2] = __byte_perm(l2, l3, 0x5410);  // row g:   inputs k+8, k+9
  a[3] = __byte_perm(l2, l3, 0x7632);  // row g+8: inputs k+8, k+9
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) mma16816(acc[M][nt], a, b[nt][2 * S], b[nt][2 * S + 1]);
}

template <int S, int NT>
__device__ __forceinline__ void kstep(const uint32_t (&w)[12], uint32_t lanebase, float (&acc)[4][NT][4],
                                      const uint32_t (&b)[NT][8]) {
  mma_step<S, 0, NT>(w, lanebase, acc, b);
  mma_step<S, 1, NT>(w, lanebase, acc, b);
  mma_step<S, 2, NT>(w, lanebase, acc, b);
  mma_step<S, 3, NT>(w, lanebase, acc, b);
}

// One super-unit: index string from the warp's ring slot, B fragments from the
// CTA's activation stage (xb = this column group's NT KB, fragment order).
template <int NT>
__device__ __forceinline__ void compute_cell(uint32_t slot, uint32_t xb, int lane, uint32_t lanebase,
                                             float (&acc)[4][NT][4]) {
  uint32_t w[12];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const uint4 v = lds128(slot + (uint32_t)(q * 512 + lane * 16));
    w[4 * q + 0] = v.x;
    w[4 * q + 1] = v.y;
    w[4 * q + 2] = v.z;
    w[4 * q + 3] = v.w;
  }
  uint32_t b[NT][8];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 v = lds128(xb + (uint32_t)((nt * 2 + h) * 512 + lane * 16));
      b[nt][4 * h + 0] = v.x;
      b[nt][4 * h + 1] = v.y;
      b[nt][4 * h + 2] = v.z;
      b[nt][4 * h + 3] = v.w;
    }
  kstep<0, NT>(w, lanebase, acc, b);
  kstep<1, NT>(w, lanebase, acc, b);
  kstep<2, NT>(w, lanebase, acc, b);
  kstep<3, NT>(w, lanebase, acc, b);
}

__device__ __forceinline__ long long range_begin(long long cells, int grid, int b) {
  return (long long)b * cells / grid;
}

// CTA owning cell x (largest b with range_begin(b) <= x).
__device__ __forceinline__ int cta_of(long long x, long long cells, int grid) {
  return (int)(((x + 1) * grid - 1) / cells);
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecArgs a) {
  constexpr int ITEMS = 16 * NT;      // accumulator values per lane
  constexpr int PIECE = 32 * ITEMS;   // floats per piece
  // dynamic shared memory: [index rings][activation stage][reduction][pad to 16 KB][2 tables]
  extern __shared__ __align__(16) unsigned char dsm[];
  const uint32_t dbase = static_cast<uint32_t>(__cvta_generic_to_shared(dsm));
  constexpr uint32_t kRingBytes = kDecWarps * Ring::kWarpBytes;
  const uint32_t xs = dbase + kRingBytes;
  float* red = reinterpret_cast<float*>(dsm + kRingBytes + Xs<NT>::kBytes);
  const uint32_t tab_off =
      ((dbase + kRingBytes + Xs<NT>::kBytes + Xs<NT>::kRedBytes + kTabAlign - 1) & ~(kTabAlign - 1)) - dbase;
  uint32_t* tabs = reinterpret_cast<uint32_t*>(dsm + tab_off);
  const uint32_t tbase = dbase + tab_off;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t ring = dbase + (uint32_t)(warp * Ring::kWarpBytes);

  // Segments (64-channel output group x matrix) form groups of S = kDecWarps/R.
  // Warp w works on segment w % S of the group and on the column groups kg with
  // kg % R == w / S; a cell is one group x one 64-input column group.
  const int R = a.ksplit, S = kDecWarps / R;
  const int seg_local = warp % S, kphase = warp / S;
  const int n_kg = a.d_in / kSuInputs;
  const int n_seg = (a.d_out / kSuChannels) * a.n_mats;
  const int n_grp = (n_seg + S - 1) / S;
  const long long cells = (long long)n_grp * n_kg;
  const long long c0 = range_begin(cells, a.grid, blockIdx.x);
  const long long c1 = range_begin(cells, a.grid, blockIdx.x + 1);
  if (c1 <= c0) return;  // uniform: no work
  if (tbase & (kTabAlign - 1)) {  // the address trick needs the 16 KB alignment; set by construction
    if (tid == 0 && a.status) atomicExch(a.status, 2);
    return;
  }

  for (int i = tid; i < kTabWords; i += kThreads) {
    tabs[i] = __ldg(a.mats[0].codebook + (i >> 5));
    if (a.n_mats > 1) tabs[kTabWords + i] = __ldg(a.mats[1].codebook + (i >> 5));
  }

  const bool two = a.n_mats > 1;
  // index prefetch cursor: the warp walks the cells of the range whose column
  // group is in its K phase, loading its own segment's super-unit of each
  long long ci = c0;
  int i_g = (int)(c0 / n_kg), i_kg = (int)(c0 % n_kg);
  auto to_phase = [&]() {
    while (ci < c1 && (i_kg & (R - 1)) != kphase) {
      ++ci;
      if (++i_kg == n_kg) {
        i_kg = 0;
        ++i_g;
      }
    }
  };
  to_phase();
  int k_issue = 0;
  auto issue = [&]() {
    const uint32_t slot = ring + (uint32_t)((k_issue % Ring::kSlots) * Ring::kSlotBytes);
    const int sg = i_g * S + seg_local;
    if (ci < c1 && sg < n_seg) {
      const int mat = two ? (sg & 1) : 0;
      const int mg = two ? (sg >> 1) : sg;
      copy_su(slot, lane, (mat ? a.mats[1].packed : a.mats[0].packed) + ((size_t)mg * n_kg + i_kg) * kSuUint4 + lane);
    }
    cp_async_commit();  // one group per cell of this warp, empty past the end
    ++k_issue;
    if (ci < c1) {
      ++ci;
      if (++i_kg == n_kg) {
        i_kg = 0;
        ++i_g;
      }
      to_phase();
    }
  };
#pragma unroll
  for (int k = 0; k < Ring::kSlots; ++k) issue();  // weights do not depend on the previous kernel
  __syncthreads();
  // Programmatic dependent launch: the above overlaps the kernel that writes the
  // rotated input; wait for it before staging activations.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  const uint4* xf_g = reinterpret_cast<const uint4*>(a.xfrag);
  int k_use = 0;
  float acc[4][NT][4];
  long long c = c0;
  while (c < c1) {
    const int g = (int)(c / n_kg);
    const long long g_end = ((long long)(g + 1) * n_kg < c1) ? (long long)(g + 1) * n_kg : c1;
    const int sg = g * S + seg_local;
    const bool live = sg < n_seg;
    const uint32_t lane_base =
        tbase | (uint32_t)(lane * 4) | ((two && (sg & 1)) ? (uint32_t)(kTabWords * 4) : 0u);
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[m][nt][j] = 0.f;

    while (c < g_end) {
      // stage the activation fragments of up to Xs<NT>::kKg column groups
      const int kA = (int)(c % n_kg);
      const int len = (int)((g_end - c) < Xs<NT>::kKg ? (g_end - c) : Xs<NT>::kKg);
      __syncthreads();  // every warp is done with the previous stage
      {
        const int per_kg = NT * 64;  // uint4 per column group
        for (int e = tid; e < len * per_kg; e += kThreads) {
          const int k = e / per_kg, r = e % per_kg;
          cp_async16(xs + (uint32_t)(e * 16), xf_g + ((size_t)(kA + k) * a.n_tiles + a.nt0) * 64 + r);
        }
        cp_async_commit();
        cp_async_wait<0>();
      }
      __syncthreads();
      for (int k = 0; k < len; ++k) {
        if (((kA + k) & (R - 1)) != kphase) continue;  // another warp's K phase
        cp_async_wait<Ring::kSlots - 1>();  // this cell's index copies have landed
        if (live)
          compute_cell<NT>(ring + (uint32_t)((k_use % Ring::kSlots) * Ring::kSlotBytes),
                           xs + (uint32_t)(k * NT * 1024), lane, lane_base, acc);
        issue();  // refill the slot just read, kSlots cells ahead
        ++k_use;
      }
      c += len;
    }
    // this CTA's part of group g: one piece per segment
    const int piece = blockIdx.x - cta_of((long long)g * n_kg, cells, a.grid);
    if (R == 1) {
      if (live) {
        float* pc = a.pieces + ((size_t)sg * a.max_pieces + piece) * PIECE;
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) pc[((m * NT + nt) * 4 + j) * 32 + lane] = acc[m][nt][j];
      }
    } else {
      // the R warps of a segment add their sums in K-phase order (deterministic)
      for (int r = 0; r < R; ++r) {
        if (kphase == r) {
          float* rd = red + seg_local * PIECE;
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int it = ((m * NT + nt) * 4 + j) * 32 + lane;
                rd[it] = (r == 0) ? acc[m][nt][j] : rd[it] + acc[m][nt][j];
              }
        }
        __syncthreads();
      }
      for (int e = tid; e < S * PIECE; e += kThreads) {
        const int sl = e / PIECE, it = e % PIECE;
        const int sg2 = g * S + sl;
        if (sg2 < n_seg) a.pieces[((size_t)sg2 * a.max_pieces + piece) * PIECE + it] = red[e];
      }
      __syncthreads();
    }
  }
}

template <int NT>
cudaError_t launch_nt(const DecArgs& a, cudaStream_t st) {
  const int dyn = kDecWarps * Ring::kWarpBytes + Xs<NT>::kBytes + Xs<NT>::kRedBytes + (int)kTabAlign + 2 * kTabWords * 4;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_kernel<NT>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_kernel<NT>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int dec_tiles_per_pass(int rows) { return rows <= 8 ? 1 : (rows <= 16 ? 2 : 4); }

// K split inside a CTA: enough warps per output segment in total (over the
// whole grid) are shared out as R warps per segment per CTA, so that each
// segment ends up with a handful of CTA pieces rather than one per warp.
int dec_ksplit(int d_in, int d_out, int n_mats) {
  const int n_seg = (d_out / kSuChannels) * n_mats;
  int sms = device_sm_count();
  if (sms > kDecMaxGrid) sms = kDecMaxGrid;
  const long long warps_per_seg = (long long)kDecWarps * sms / n_seg;
  int r = 1;
  while (r < kDecWarps && 2LL * r * 3 <= warps_per_seg) r *= 2;
  const int n_kg = d_in / kSuInputs;
  while (r > 1 && r > n_kg) r /= 2;
  return r;
}

int dec_groups(int d_in, int d_out, int n_mats) {
  const int n_seg = (d_out / kSuChannels) * n_mats;
  const int s = kDecWarps / dec_ksplit(d_in, d_out, n_mats);
  return (n_seg + s - 1) / s;
}

int dec_grid(int d_in, int d_out, int n_mats) {
  int g = device_sm_count();
  if (g > kDecMaxGrid) g = kDecMaxGrid;
  const long long cells = (long long)dec_groups(d_in, d_out, n_mats) * (d_in / kSuInputs);
  return cells < g ? (int)cells : g;  // every CTA owns at least one cell
}

int dec_max_pieces(int d_in, int d_out, int n_mats, int grid) {
  const long long n_kg = d_in / kSuInputs;
  const long long n_grp = dec_groups(d_in, d_out, n_mats);
  const long long cells = n_grp * n_kg;
  int best = 1;
  for (long long s = 0; s < n_grp; ++s) {
    const long long x0 = s * n_kg, x1 = x0 + n_kg - 1;
    const long long b0 = ((x0 + 1) * grid - 1) / cells, b1 = ((x1 + 1) * grid - 1) / cells;
    if (b1 - b0 + 1 > best) best = (int)(b1 - b0 + 1);
  }
  return best;
}

cudaError_t launch_decode(const DecArgs& a, int nt, cudaStream_t st) {
  switch (nt) {
    case 1: return launch_nt<1>(a, st);
    case 2: return launch_nt<2>(a, st);
    case 4: return launch_nt<4>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vq3
