// The many-row path (prefill, T >= 64) of the VQ3 matrices: a tensor-core GEMM
// on 5th-generation tensor cores (tcgen05) whose weight operand is decoded from
// the three-bit vector LUT on the fly.
//
// What it computes (model card "anemll/anemll-forge-qwen3.8-27B", section
// "Release 0.2: three-bit MLP, token-mixer rotations, distilled weights": a 2x64
// vector LUT per matrix, one six-bit index per output pair and input, per-channel
// scales; SiLU per "ANEMLL ANE LLM conversion pipeline", "Facts"), for activations
// already rotated (x' = R x, in FP16):
//   linear / down:  y[r][o] = fp16( s[o] * sum_i W0[o][i] x'[r][i] ),  W0[2p+c][i] = C[idx[p][i]][c]
//   gate + up:      h[r][j] = silu(s_g[j] g[r][j]) * (s_u[j] u[r][j])  (FP32)
//
// An output tile is 128 channels x N rows (N <= 256), its FP32 accumulator
// D[channel][row] in tensor memory, summed over K in steps of 64 inputs (one column
// group of the packed super-units). The work is a persistent stream-K split of the (tile, K step) space: each CTA takes a
// contiguous run of steps; a tile split between CTAs is summed in K order by the CTA
// holding its first steps, from the raw partial sums of the others (per-CTA flags).
//   warp 0     lane 0 issues, per K step, the TMA copy of the activation tile B[N][64]
//              (128-byte swizzle, rows past the last read as zeros), the bulk copies of
//              the two super-units of index strings, and an L2 prefetch of the index
//              strings a few steps further on, all completing on the step's load barrier.
//   warps 1-8  decoders: once a step's index strings are in, each warp takes part of the
//              lane strings of one super-unit, looks the indices up in a lane-private
//              shared-memory copy of the codebook and pairs neighbouring inputs of a
//              channel with a byte permute into the FP16 words of A[128][64], in the
//              K-major "core matrix" layout (8 rows x 16 bytes per 128-byte block) that
//              the MMA's shared-memory descriptors read.
//   warp 9     one lane issues tcgen05.mma (M = 128, N, K = 16) four times per K step;
//              tcgen05.commit releases the step's load stage and A tile, and at the end
//              of a tile marks its accumulator (one of two in tensor memory) complete.
//   warps 10-13 epilogue: tcgen05.ld of the accumulator (each warp its 32 lanes), the
//              later parts of a split tile, scale (and SwiGLU: the tile's rows 0-63 are
//              gate channels, rows 64-127 the up channels of the same 64) and store.
// Two mbarrier rings connect them: load stages (B tile + index strings; as many as fit,
// so that copies run far ahead) and decoded A tiles (two or three). All waits are
// bounded: one that runs out sets the status word to 3 and the kernel carries on to its
// end (results invalid).
#include <cuda.h>  // CUtensorMap; the encoder is fetched from the driver at run time
#include <cuda_fp16.h>

#include <utility>

#include "vq3_internal.h"

namespace vq3 {
VQ3_BOUNDS_RECORD(prefill_wide)
namespace {

constexpr int kTmaWarp = 0;                     // lane 0 issues the tile copies
constexpr int kDecWarp0 = 1;
constexpr int kDecWarps = 8;                    // warps 1-8
constexpr int kMmaWarp = kDecWarp0 + kDecWarps;  // 9
constexpr int kEpiWarp0 = kMmaWarp + 1;          // warps 10-13
constexpr int kPThreads = (kEpiWarp0 + 4) * 32;
constexpr int kEpiThreads = 4 * 32;
constexpr int kMinSteps = 8;  // fewest K steps per CTA
constexpr int kMaxStages = 12;  // load stages
constexpr int kMaxAStages = 3;  // decoded A tiles
constexpr int kPrefetchSteps = 8;  // index strings are prefetched into L2 this many K steps ahead
constexpr int kTileM = 128;                    // output channels per tile
constexpr int kATile = kTileM * 64 * 2;        // 16 KB of FP16
// Lane-private codebook tables (entry k of lane L at word k*32 + L), the gate and
// up tables kStride bytes apart and aligned to twice that (matrix choice by OR).
template <int F>
struct PfTab {
  static constexpr uint32_t kStride = (uint32_t)Fmt<F>::kEntries * 128u;
  static constexpr uint32_t kAlign = 2u * kStride;
};
constexpr unsigned long long kWaitNs = 1000000000ull;  // a wait gives up after one second
constexpr unsigned long long kDrainNs = 100000000ull;  // the end-of-kernel drain waits at most 0.1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `parity` to complete, bounded in time. `abort` is the
// CTA's shared flag: once set (a wait of this CTA gave up, or another CTA's did: status
// word 3, read every 256 polls) every wait returns at once. A wait that runs past kWaitNs
// sets the status word to 3 and the flag.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, int* status, volatile int* abort) {
  if (mbar_try_wait(bar, parity) || *abort) return;
  const unsigned long long t0 = globaltimer_ns();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity) || *abort) return;
    if ((it & 255u) == 0u) {
      if (*(volatile int*)status == 3) {
        *abort = 1;
        return;
      }
      if (globaltimer_ns() - t0 > kWaitNs) {
        atomicExch(status, 3);
        *abort = 1;
        return;
      }
    }
  }
}

// End-of-kernel drain: wait (at most kDrainNs, whatever the abort flag says) for a phase
// whose asynchronous work was issued, so that no copy or MMA is in flight at exit.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kDrainNs) return;
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Tile (x, y) of a 2D tensor map into shared memory; completes `bytes` of the barrier's transaction count.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Brings a contiguous global range (16-byte aligned, a multiple of 16 bytes) into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Contiguous global -> shared copy (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand without swizzle: core
// matrices of 8 rows x 16 bytes stored as 128 contiguous bytes; lbo = byte step
// between core matrices along K, sbo = byte step along M/N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// The same for a K-major operand in the 128-byte swizzle layout: rows of 64 FP16
// (128 bytes), 8-row atoms of 1 KB (sbo), the 16-byte chunk c of row r stored at
// chunk position c ^ (r % 8); the atoms are 1 KB aligned. K advances inside an
// atom by moving the start address (32 bytes per 16 elements).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                    // leading byte offset: unused with this swizzle
  d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset: one 8-row atom
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with FP16 A and B, FP32 D, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Lookup address of index N of a lane string: bits [b N, b N + b) (b = index
// width) moved to [7, 7 + b) (entry stride 32 lanes x 4 bytes), OR-ed with the
// table base and lane column.
template <int F, int N>
__device__ __forceinline__ uint32_t lut_addr(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase) {
  constexpr int kB = Fmt<F>::kBits;
  constexpr int pos = kB * N, wd = pos >> 5, off = pos & 31;
  constexpr uint32_t mask = ((1u << kB) - 1u) << 7;
  uint32_t v;
  if constexpr (off + kB > 32) {
    v = __funnelshift_r(w[wd], w[wd + 1], off - 7);  // the field straddles two words
  } else if constexpr (off >= 7) {
    v = w[wd] >> (off - 7);
  } else {
    v = w[wd] << (7 - off);
  }
  return (v & mask) | lanebase;
}

// Byte offset of (row, k) in a K-major core-matrix tile with `rows` rows and 64
// columns of K: core matrix (row/8, k/8) at (k/8) * rows * 16 + (row/8) * 128.
__device__ __forceinline__ uint32_t tile_off(int row, int k, int rows) {
  return (uint32_t)((k >> 3) * rows * 16 + (row >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

template <int F, int N0, int NL, int... J>
__device__ __forceinline__ void lookups(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase, uint32_t (&lk)[NL],
                                        std::integer_sequence<int, J...>) {
  ((lk[J] = lds32(lut_addr<F, N0 + J>(w, lanebase))), ...);
}

// Decodes the producer thread's share of the weight tile of one K step: input
// steps S0 .. S0 + NS - 1 (16 inputs each) of lane string L = lane of one
// super-unit. Lane-string order (see vq3_internal.h): for the vector formats
// index n = (s*4 + m)*4 + e is pair m*8 + g at input s*16 + {2t, 2t+1, 2t+8,
// 2t+9}[e]; for the scalar format index 2n + c is channel 2(m*8 + g) + c at the
// same input; g = L/4, t = L%4. All lookups are issued before the first store,
// so one shared-memory latency covers them. Channels 2p and 2p+1 of a pair are
// 16 bytes apart in the tile; lanes with g >= 4 store the odd channel first,
// which puts the 32 lanes of each store on 32 different banks.
template <int F, int S0, int NS>
__device__ __forceinline__ void decode_steps(const uint32_t (&w)[Fmt<F>::kWords], int lane, int row0,
                                             uint32_t a_tile, uint32_t lanebase) {
  constexpr int kPerStep = 32 / Fmt<F>::kVec;  // lookups per k-step of 16 inputs: 16 (vector) or 32 (scalar)
  uint32_t lk[kPerStep * NS];
  lookups<F, S0 * kPerStep, kPerStep * NS>(w, lanebase, lk, std::make_integer_sequence<int, kPerStep * NS>{});
  const int g = lane >> 2, t = lane & 3;
  const bool odd_first = g >= 4;
  const uint32_t swap = odd_first ? 16u : 0u;
  const uint32_t sel_a = odd_first ? 0x7632u : 0x5410u, sel_b = sel_a ^ 0x2222u;
#pragma unroll
  for (int sm = 0; sm < 4 * NS; ++sm) {  // (s - S0, m)
    const int S = S0 + (sm >> 2), M = sm & 3;
    const int r = row0 + 2 * (M * 8 + g);  // channel 2p of the tile; 2p+1 is the next row
    const int k = S * 16 + 2 * t;
    const uint32_t o0 = a_tile + tile_off(r, k, kTileM), o8 = a_tile + tile_off(r, k + 8, kTileM);
    if constexpr (Fmt<F>::kVec == 2) {
      const uint32_t* l = lk + 4 * sm;
      sts32(o0 + swap, __byte_perm(l[0], l[1], sel_a));
      sts32(o0 + (16u - swap), __byte_perm(l[0], l[1], sel_b));
      sts32(o8 + swap, __byte_perm(l[2], l[3], sel_a));
      sts32(o8 + (16u - swap), __byte_perm(l[2], l[3], sel_b));
    } else {
      const uint32_t* l = lk + 8 * sm;  // index (e, c) at 2e + c
      const uint32_t a0 = __byte_perm(l[0], l[2], 0x5410), a1 = __byte_perm(l[1], l[3], 0x5410);
      const uint32_t a2 = __byte_perm(l[4], l[6], 0x5410), a3 = __byte_perm(l[5], l[7], 0x5410);
      sts32(o0 + swap, odd_first ? a1 : a0);
      sts32(o0 + (16u - swap), odd_first ? a0 : a1);
      sts32(o8 + swap, odd_first ? a3 : a2);
      sts32(o8 + (16u - swap), odd_first ? a2 : a3);
    }
  }
}

// Decoder warps per super-unit and input steps per warp.
constexpr int kDecPerSu = kDecWarps / 2;
constexpr int kStepsPerDec = 4 / kDecPerSu;
static_assert(kDecWarps == 2 || kDecWarps == 4 || kDecWarps == 8, "decoder warps split the 4 input steps evenly");

template <int F>
__device__ __forceinline__ void decode_part(const uint32_t (&w)[Fmt<F>::kWords], int part, int lane, int row0,
                                            uint32_t a_tile, uint32_t lanebase) {
  if constexpr (kStepsPerDec == 1) {
    switch (part) {
      case 0: decode_steps<F, 0, 1>(w, lane, row0, a_tile, lanebase); break;
      case 1: decode_steps<F, 1, 1>(w, lane, row0, a_tile, lanebase); break;
      case 2: decode_steps<F, 2, 1>(w, lane, row0, a_tile, lanebase); break;
      default: decode_steps<F, 3, 1>(w, lane, row0, a_tile, lanebase); break;
    }
  } else if constexpr (kStepsPerDec == 2) {
    if (part == 0)
      decode_steps<F, 0, 2>(w, lane, row0, a_tile, lanebase);
    else
      decode_steps<F, 2, 2>(w, lane, row0, a_tile, lanebase);
  } else {
    decode_steps<F, 0, 4>(w, lane, row0, a_tile, lanebase);
  }
}

template <int N, int F>
struct PfSmem {
  static constexpr int kBTile = N * 64 * 2;
  static constexpr int kSu = FmtSizes<F>::kSuBytes;
  static constexpr int kIdxBytes = 2 * kSu;  // index strings of the tile's two super-units per K step
  static constexpr int kLoadBytes = kBTile + kIdxBytes;
  static_assert(kBTile % 1024 == 0 && kATile % 1024 == 0, "B tiles start on 1 KB swizzle atoms");
  // alignment slack of the stage area, codebook tables (with their alignment slack), SwiGLU
  // exchange; and room for the kernel's static shared memory
  static constexpr int kFixed = 1024 + (int)PfTab<F>::kAlign + 2 * (int)PfTab<F>::kStride + 64 * 16 * 4;
  static constexpr int kStaticRoom = 512;
  // Decoded A tiles in flight: the decoders run ahead of the MMA by kAStages - 1 steps.
  static constexpr int kAStages = N >= 256 ? 2 : 3;
  // Load stages (B tile and index strings): as many as fit. The K loop is bound by the round
  // trip from a stage's MMA completion through its refill to its next MMA, so the load ring,
  // not the A tiles, sets how many steps are in flight.
  static constexpr int kFit = (227 * 1024 - kStaticRoom - kFixed - kAStages * kATile) / kLoadBytes;
  static constexpr int kLoadStages = kFit > kMaxStages ? kMaxStages : kFit;
  static_assert(kLoadStages >= 2 && kAStages <= kMaxAStages, "stage counts");
  static constexpr int kBOffset = kAStages * kATile;                 // B tiles
  static constexpr int kIOffset = kBOffset + kLoadStages * kBTile;   // index strings
  static constexpr int kStageArea = kIOffset + kLoadStages * kIdxBytes;
  static constexpr int kTotal = kFixed + kStageArea;
  static_assert(kTotal + kStaticRoom <= 227 * 1024, "shared memory per CTA");
};

// This CTA's share of the (tile, K step) space: steps [begin(c), begin(c + 1)).
__host__ __device__ __forceinline__ long long range_begin(int c, long long work, int grid) {
  return work * c / grid;
}

// One segment of a CTA's range: K steps [k0, k1) of tile t.
struct Seg {
  int t, k0, k1;
};
__device__ __forceinline__ Seg seg_at(long long s, long long s1, int n_kg) {
  Seg g;
  g.t = (int)(s / n_kg);
  g.k0 = (int)(s - (long long)g.t * n_kg);
  const long long left = s1 - s;
  g.k1 = left < (long long)(n_kg - g.k0) ? g.k0 + (int)left : n_kg;
  return g;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One CTA per SM: the smallest configuration still needs more than half of an
// SM's shared memory, so no two CTAs ever share an SM (and its tensor memory).
static_assert(2 * PfSmem<64, VQ3_FORMAT_2X16>::kTotal > 228 * 1024, "one prefill CTA per SM");

template <int N, int F>
__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(const __grid_constant__ PrefillArgs a,
                                                                     const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ __align__(16) unsigned char dsm[];
  using PS = PfSmem<N, F>;
  constexpr int kSL = PS::kLoadStages, kSA = PS::kAStages;
  __shared__ __align__(8) unsigned long long s_bars[2 * kMaxStages + 2 * kMaxAStages + 5];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;  // set once a wait of this CTA gave up or saw status 3
  volatile int* abort = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = smem_u32(dsm);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 1 KB aligned stages (swizzle atoms)
  const uint32_t tabs = (base + PS::kStageArea + PfTab<F>::kAlign - 1) & ~(PfTab<F>::kAlign - 1);
  float* xch = reinterpret_cast<float*>(dsm + (tabs - raw) + 2 * PfTab<F>::kStride);  // up values for SwiGLU
  const uint32_t bar0 = smem_u32(s_bars);
  auto load_full = [&](int s) { return bar0 + 8u * s; };                       // B and indices landed
  auto load_empty = [&](int s) { return bar0 + 8u * (kSL + s); };              // B and indices consumed
  auto a_full = [&](int s) { return bar0 + 8u * (2 * kSL + s); };              // A decoded
  auto a_empty = [&](int s) { return bar0 + 8u * (2 * kSL + kSA + s); };       // A consumed
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kSL + 2 * kSA + b); };  // accumulator b complete
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kSL + 2 * kSA + 2 + b); };  // accumulator b drained
  const uint32_t mma_drain = bar0 + 8u * (2 * kSL + 2 * kSA + 4);              // every MMA issued has completed
  auto a_tile = [&](int s) { return base + (uint32_t)(s * kATile); };
  auto b_tile = [&](int s) { return base + (uint32_t)(PS::kBOffset + s * PS::kBTile); };
  auto i_tile = [&](int s) { return base + (uint32_t)(PS::kIOffset + s * PS::kIdxBytes); };

  const int n_kg = a.d_in / 64;
  const int n_tiles = (a.rows + N - 1) / N;  // row tiles
  const long long s0 = range_begin(blockIdx.x, a.work, gridDim.x);
  const long long s1 = range_begin(blockIdx.x + 1, a.work, gridDim.x);

  // codebook tables (lane-private copies): matrix 0 at tabs, matrix 1 one stride on; a
  // vector entry is (component 0 | component 1 << 16), a scalar one (entry | entry << 16)
  constexpr int E = Fmt<F>::kEntries;
  for (int i = tid; i < 2 * E * 8; i += kPThreads) {
    const int t2 = i / (E * 8), k = (i >> 3) % E, q = i & 7;
    const uint32_t* cb = t2 ? a.cb1 : a.cb0;
    if (cb) {
      uint32_t v;
      if constexpr (Fmt<F>::kVec == 2) {
        v = __ldg(cb + k);
      } else {
        const uint32_t h = __ldg(reinterpret_cast<const uint16_t*>(cb) + k);
        v = h | (h << 16);
      }
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                       tabs + (uint32_t)(t2 * PfTab<F>::kStride + k * 128 + q * 16)),
                   "r"(v)
                   : "memory");
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kSL; ++s) {
      mbar_init(load_full(s), 1);
      mbar_init(load_empty(s), 1);
    }
    for (int s = 0; s < kSA; ++s) {
      mbar_init(a_full(s), kDecWarps * 32);
      mbar_init(a_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kEpiThreads);
    }
    mbar_init(mma_drain, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"((uint32_t)(2 * N))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ tile copies
    if (lane == 0) {
      constexpr uint32_t kTx = (uint32_t)(PS::kBTile + PS::kIdxBytes);
      constexpr int kSuU4 = FmtSizes<F>::kSuUint4;
      constexpr uint32_t kSuB = (uint32_t)PS::kSu;
      int it = 0;
      for (long long s = s0; s < s1;) {
        const Seg g = seg_at(s, s1, n_kg);
        const int mt = g.t / n_tiles, row0 = (g.t - mt * n_tiles) * N;
        // the tile's two super-units: (matrix, channel group); the second is past the
        // last channel when d_out is an odd multiple of 64 (its A rows are never stored)
        const int mg0 = a.swiglu ? mt : 2 * mt, mg1 = a.swiglu ? mt : 2 * mt + 1;
        const bool live1 = a.swiglu || mg1 < a.d_out / 64;
        const uint4* su0 = a.packed0 + (size_t)mg0 * n_kg * kSuU4;
        const uint4* su1 = (a.swiglu ? a.packed1 : a.packed0) + (size_t)(live1 ? mg1 : mg0) * n_kg * kSuU4;
        for (int kk = g.k0; kk < g.k1 && !*abort; ++kk, ++it) {
          const int ls = it % kSL;
          if (it >= kSL) mbar_wait(load_empty(ls), (uint32_t)((it / kSL - 1) & 1), a.status, abort);
          if (*abort) break;  // a wait gave up: no further copies
          mbar_expect_tx(load_full(ls), kTx);
          // activation tile: N rows x 64 inputs in the 128-byte swizzle layout (rows
          // past the last are filled with zeros)
          if (kk + kPrefetchSteps < g.k1) {
            prefetch_l2(su0 + (size_t)(kk + kPrefetchSteps) * kSuU4, kSuB);
            prefetch_l2(su1 + (size_t)(kk + kPrefetchSteps) * kSuU4, kSuB);
          }
          tma_load_2d(b_tile(ls), &xmap, kk * 64, row0, load_full(ls));
          bulk_load(i_tile(ls), su0 + (size_t)kk * kSuU4, kSuB, load_full(ls));
          bulk_load(i_tile(ls) + kSuB, su1 + (size_t)kk * kSuU4, kSuB, load_full(ls));
        }
        s += g.k1 - g.k0;
      }
      // steps [0, it) were issued: wait for the copies of the last use of each stage to land
      // (done long ago unless a wait gave up), so that none is in flight at exit
      for (int j = it > kSL ? it - kSL : 0; j < it; ++j) mbar_drain(load_full(j % kSL), (uint32_t)((j / kSL) & 1));
    }
    __syncwarp();
  } else if (warp < kDecWarp0 + kDecWarps) {
    // ------------------------------------------------------------ decoders
    // warp -> (super-unit su of the tile, part of the lane strings); lane -> lane string
    const int dw = warp - kDecWarp0;
    const int su = dw / kDecPerSu, part = dw % kDecPerSu, L = lane;
    const int s_lo = part * kStepsPerDec, s_hi = s_lo + kStepsPerDec;  // input steps of this warp
    const uint32_t lanebase = tabs | (uint32_t)(lane * 4) | ((a.swiglu && su == 1) ? PfTab<F>::kStride : 0u);
    int it = 0;
    for (long long s = s0; s < s1;) {
      const Seg g = seg_at(s, s1, n_kg);
      const int mt = g.t / n_tiles;
      const bool live = su == 0 || a.swiglu || 2 * mt + 1 < a.d_out / 64;
      for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
        const int ls = it % kSL, as = it % kSA;
        if (it >= kSA) mbar_wait(a_empty(as), (uint32_t)((it / kSA - 1) & 1), a.status, abort);
        mbar_wait(load_full(ls), (uint32_t)((it / kSL) & 1), a.status, abort);
        if (live) {
          // input steps [s_lo, s_hi) are words kW s_lo .. kW s_hi of the string (kW
          // words per step; the last word for six-bit indices that straddle two)
          constexpr int kW = Fmt<F>::kWords / 4;
          uint32_t w[Fmt<F>::kWords] = {};
          const uint32_t is = i_tile(ls) + (uint32_t)(su * PS::kSu);
#pragma unroll
          for (int q = 0; q < FmtSizes<F>::kChunks; ++q) {
            if (4 * q > kW * s_hi || 4 * q + 3 < kW * s_lo) continue;
            const uint32_t o = is + (uint32_t)((q * 32 + L) * 16);
            uint32_t v0, v1, v2, v3;
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3) : "r"(o));
            w[4 * q + 0] = v0;
            w[4 * q + 1] = v1;
            w[4 * q + 2] = v2;
            w[4 * q + 3] = v3;
          }
          decode_part<F>(w, part, L, su * 64, a_tile(as), lanebase);
        }
        fence_proxy_async();  // the generic-proxy writes of A, before the MMA reads them
        mbar_arrive(a_full(as));
      }
      s += g.k1 - g.k0;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTileM, N);
      int it = 0, q = 0;
      for (long long s = s0; s < s1; ++q) {
        const Seg g = seg_at(s, s1, n_kg);
        const int b = q & 1;
        if (q >= 2) mbar_wait(acc_empty(b), (uint32_t)(((q >> 1) - 1) & 1), a.status, abort);
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(b * N);
        for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
          const int ls = it % kSL, as = it % kSA;
          mbar_wait(load_full(ls), (uint32_t)((it / kSL) & 1), a.status, abort);
          mbar_wait(a_full(as), (uint32_t)((it / kSA) & 1), a.status, abort);
          if (*abort) continue;  // a wait gave up: no further MMAs (the consumers return at once)
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // K = 16: two core matrices along K
            const uint64_t ad = smem_desc(a_tile(as) + (uint32_t)(j * 2 * kTileM * 16), kTileM * 16, 128);
            const uint64_t bd = smem_desc_sw128(b_tile(ls) + (uint32_t)(j * 32));
            mma_ss(acc, ad, bd, idesc, (kk > g.k0 || j > 0) ? 1u : 0u);
          }
          mma_commit(load_empty(ls));  // both complete when this step's MMAs have read their operands
          mma_commit(a_empty(as));
        }
        mma_commit(acc_full(b));
        s += g.k1 - g.k0;
      }
      // every MMA issued has completed before the tensor memory is freed (at once unless a
      // wait gave up and the epilogue stopped waiting for the accumulators)
      mma_commit(mma_drain);
      mbar_drain(mma_drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // TMEM lanes 32*(warp % 4) .. +31 = tile rows = output channels of the tile
    const int row = (warp & 3) * 32 + lane;
    const int e = tid - kEpiWarp0 * 32;
    const bool waits = *(volatile int*)a.status == 0;
    int q = 0;
    for (long long s = s0; s < s1; ++q) {
      const Seg g = seg_at(s, s1, n_kg);
      const int mt = g.t / n_tiles, row0 = (g.t - mt * n_tiles) * N;
      const int cols = a.rows - row0 < N ? a.rows - row0 : N;  // valid rows of this tile
      const int b = q & 1;
      mbar_wait(acc_full(b), (uint32_t)((q >> 1) & 1), a.status, abort);
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)(b * N) + ((uint32_t)((warp & 3) * 32) << 16);
      if (g.k0 > 0) {
        // a later part of a tile started by an earlier CTA: hand the raw sums over
        float* part = a.part + (size_t)blockIdx.x * kTileM * N;
#pragma unroll 1
        for (int c0 = 0; c0 < cols; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(taddr + (uint32_t)c0, r);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (VQ3_IN((size_t)blockIdx.x * kTileM * N + (size_t)(c0 + j) * kTileM + row, (size_t)gridDim.x * kTileM * N, 1))
              __stcg(part + (size_t)(c0 + j) * kTileM + row, __uint_as_float(r[j]));
        }
        tc_fence_before();
        mbar_arrive(acc_empty(b));
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (e == 0) asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a.flags + blockIdx.x), "r"(1u) : "memory");
      } else {
        // the tile's first part: add the later parts (CTAs blockIdx.x + 1 ...) in K order
        int n_parts = 0;
        if (g.k1 < n_kg) {
          const long long tile_end = (long long)(g.t + 1) * n_kg;
          while ((int)blockIdx.x + 1 + n_parts < (int)gridDim.x &&
                 range_begin(blockIdx.x + 1 + n_parts, a.work, gridDim.x) < tile_end)
            ++n_parts;
          if (e == 0 && waits) {
            for (int p = 1; p <= n_parts && !*abort; ++p) {
              if (!VQ3_IN(blockIdx.x + p, gridDim.x, 2)) break;
              const unsigned long long t0 = globaltimer_ns();
              for (unsigned spin = 1; ld_acquire_u32(a.flags + blockIdx.x + p) == 0u && !*abort; ++spin) {
                __nanosleep(64);
                if ((spin & 255u) == 0u && globaltimer_ns() - t0 > kWaitNs) {
                  atomicExch(a.status, 3);
                  *abort = 1;
                }
              }
            }
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        const float* parts = a.part + (size_t)(blockIdx.x + 1) * kTileM * N;
        if (!a.swiglu) {
          const int ch = mt * kTileM + row;
          const bool live = ch < a.d_out;
          const float sc = live ? __half2float(__ushort_as_half(a.scale0[ch])) : 0.f;
#pragma unroll 1
          for (int c0 = 0; c0 < cols; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + (uint32_t)c0, r);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
            for (int p = 0; p < n_parts; ++p) {
              if (!VQ3_IN((size_t)(blockIdx.x + 1 + p) * kTileM * N + (size_t)(c0 + 15) * kTileM + row,
                          (size_t)gridDim.x * kTileM * N, 3))
                break;
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] += __ldcg(parts + (size_t)p * kTileM * N + (size_t)(c0 + j) * kTileM + row);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] *= sc;
            if (a.lr_y && live) {
              // low-rank correction, one value per output (lanes: consecutive channels)
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < cols && VQ3_IN((size_t)(row0 + c0 + j) * a.d_out + ch, (size_t)a.rows * a.d_out, 4))
                  v[j] += __ldg(a.lr_y + (size_t)(row0 + c0 + j) * a.d_out + ch);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int rr = row0 + c0 + j;
              if (live && c0 + j < cols && VQ3_IN((size_t)rr * a.d_out + ch, (size_t)a.rows * a.d_out, 5))
                a.out16[(size_t)rr * a.d_out + ch] = __half_as_ushort(__float2half_rn(v[j]));
            }
          }
        } else {
          // rows 0-63: gate channel mt*64 + row; rows 64-127: up channel mt*64 + row - 64
          const int jch = mt * 64 + (row & 63);
          const bool up = row >= 64;
          const float sc = __half2float(__ushort_as_half(up ? a.scale1[jch] : a.scale0[jch]));
#pragma unroll 1
          for (int c0 = 0; c0 < cols; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + (uint32_t)c0, r);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
            for (int p = 0; p < n_parts; ++p) {
              if (!VQ3_IN((size_t)(blockIdx.x + 1 + p) * kTileM * N + (size_t)(c0 + 15) * kTileM + row,
                          (size_t)gridDim.x * kTileM * N, 3))
                break;
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] += __ldcg(parts + (size_t)p * kTileM * N + (size_t)(c0 + j) * kTileM + row);
            }
            if (up) {
#pragma unroll
              for (int j = 0; j < 16; ++j) xch[j * 64 + (row - 64)] = sc * v[j];
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (!up) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int rr = row0 + c0 + j;
                const float hv = silu_f(sc * v[j]) * xch[j * 64 + row];
                if (c0 + j < cols && VQ3_IN((size_t)rr * a.d_out + jch, (size_t)a.rows * a.d_out, 6))
                  __stcg(a.out32 + (size_t)rr * a.d_out + jch, hv);
              }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
          }
        }
        tc_fence_before();
        mbar_arrive(acc_empty(b));
        if (n_parts) {
          // every epilogue thread has read the parts: their flags go back to zero
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (e == 0)
            for (int p = 1; p <= n_parts; ++p) a.flags[blockIdx.x + p] = 0u;
        }
      }
      s += g.k1 - g.k0;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)(2 * N))
                 : "memory");
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      p = nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// The activations [rows][d_in] FP16 as tiles of 64 inputs x N rows in the
// 128-byte swizzle layout; rows past the last read as zeros.
cudaError_t activation_map(const PrefillArgs& a, int n, CUtensorMap* map) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)a.d_in, (cuuint64_t)a.rows};
  const cuuint64_t strides[1] = {(cuuint64_t)a.d_in * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)n};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(a.x), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int N, int F>
cudaError_t launch_n(PrefillArgs a, cudaStream_t st) {
  const int smem = PfSmem<N, F>::kTotal;
  cudaError_t e = cudaFuncSetAttribute(prefill_gemm_kernel<N, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap xmap;
  if ((e = activation_map(a, N, &xmap)) != cudaSuccess) return e;
  a.work = prefill_wide_work(a.rows, a.d_in, a.d_out, a.swiglu);
  const int grid = prefill_wide_grid(a.rows, a.d_in, a.d_out, a.swiglu);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the first part of a split tile waits for the others
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<N, F>, a, xmap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

long long prefill_wide_work(int rows, int d_in, int d_out, int swiglu) {
  const long long m_tiles = swiglu ? d_out / 64 : (d_out + kTileM - 1) / kTileM;
  return m_tiles * ((rows + 255) / 256) * (d_in / 64);
}

int prefill_wide_grid(int rows, int d_in, int d_out, int swiglu) {
  const long long work = prefill_wide_work(rows, d_in, d_out, swiglu);
  const long long g = work / kMinSteps;
  const int cap = device_sm_count();
  return g < 1 ? 1 : (g < cap ? (int)g : cap);
}

namespace {
template <int F>
cudaError_t launch_fmt(const PrefillArgs& a, cudaStream_t st) {
  return launch_n<256, F>(a, st);
}
}  // namespace

cudaError_t launch_prefill_wide_gemm(const PrefillArgs& a, cudaStream_t st) {
  switch (a.format) {
    case VQ3_FORMAT_2X64: return launch_fmt<VQ3_FORMAT_2X64>(a, st);
    case VQ3_FORMAT_2X16: return launch_fmt<VQ3_FORMAT_2X16>(a, st);
    case VQ3_FORMAT_LUT4: return launch_fmt<VQ3_FORMAT_LUT4>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vq3
