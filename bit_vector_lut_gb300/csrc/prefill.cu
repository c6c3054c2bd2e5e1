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
// bounded in time: one that runs out sets the status word to 3 and the CTA's abort flag,
// after which no copy or MMA is issued and every wait returns at once; before the tensor
// memory is freed the copy thread waits for its copies in flight and the MMA thread for
// its MMAs (each drain bounded too), and the kernel ends (results invalid).
#include <cuda.h>  // CUtensorMap; the encoder is fetched from the driver at run time
#include <cuda_fp16.h>

#include <utility>

#include "vq3_internal.h"

namespace vq3 {
VQ3_BOUNDS_RECORD(prefill)
namespace {

constexpr int kTmaWarp = 0;                     // lane 0 issues the tile copies
constexpr int kDecWarp0 = 1;
constexpr int kDecWarps = 16;                   // warps 1-16, four per tensor-memory lane quarter
constexpr int kMmaWarp = kDecWarp0 + kDecWarps;  // 17
constexpr int kEpiWarp0 = kMmaWarp + 1;          // warps 18-21
constexpr int kPThreads = (kEpiWarp0 + 4) * 32;
constexpr int kEpiThreads = 4 * 32;
constexpr int kMinSteps = 8;  // fewest K steps per CTA
constexpr int kMaxStages = 8;  // load stages
constexpr int kMaxAStages = 3;  // decoded A stages in tensor memory (one step's G tiles each)
constexpr int kPrefetchSpan = 8;  // index strings go to L2 in spans of this many K steps, one span ahead
constexpr int kTileM = 128;                    // output channels per tile
constexpr int kTileCols = 256;                 // accumulator columns per step: G tiles x N rows
constexpr int kTmemCols = 512;                 // tensor memory: accumulators, then the decoded A stages
constexpr int kACols = 32;                     // one decoded A tile (128 lanes x 64 FP16 inputs)
constexpr int kMaxGrid = 256;                  // most CTAs of one launch (the launcher caps the grid)
// Lane-private codebook tables (entry k of lane L at word k*32 + L), the gate and
// up tables kStride bytes apart, each aligned to kStride (the lookup ORs the lane's
// column and the entry into the table's address).
template <int F>
struct PfTab {
  static constexpr uint32_t kStride = (uint32_t)Fmt<F>::kEntries * 128u;
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
// Box (x, y, z, w) of a 4D tensor map into shared memory (x a multiple of 16 bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
// Brings a contiguous global range (16-byte aligned, a multiple of 16 bytes) into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand in the 128-byte swizzle layout: rows of 64 FP16
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

// The four K = 16 MMAs of one K step (64 inputs) of one tile, from one elected lane:
// A columns a_tmem + 0, 8, 16, 24 (tensor memory), B descriptors bdesc + 0, 2, 4, 6 (32
// bytes further along the swizzled rows each); the first accumulates only if acc != 0.
__device__ __forceinline__ void mma_ts_kstep(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q, e;\n .reg .b32 a1, a2, a3;\n .reg .b64 b1, b2, b3;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 q, %4, %4;\n"
      " add.u32 a1, %1, 8;\n add.u32 a2, %1, 16;\n add.u32 a3, %1, 24;\n"
      " add.u64 b1, %2, 2;\n add.u64 b2, %2, 4;\n add.u64 b3, %2, 6;\n"
      " elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, q;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, q;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, q;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// tcgen05.commit from one elected lane of a converged warp.
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
      : "memory");
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

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void tmem_st16x256(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

// The lane's part of 16-channel tile M x 16-input step S of a decoded A tile, in the
// register order of tcgen05.st 16x256b: r[0] (lane g, column 2t), r[1] (lane g, column
// 2t+1), r[2] (lane g+8, column 2t), r[3] (lane g+8, column 2t+1), with TMEM lane g the
// pair's channel 2p and lane g+8 its channel 2p+1 (p = 8M + g), column 2t the inputs
// 2t, 2t+1 of the step and column 2t+1 the inputs 2t+8, 2t+9 (the operand order of
// mma_order_col). g = lane / 4, t = lane % 4, as in the lane strings.
template <int F, int S, int M>
__device__ __forceinline__ void tmem_frag(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase, uint32_t (&r)[4]) {
  if constexpr (Fmt<F>::kVec == 2) {
    constexpr int n0 = (S * 4 + M) * 4;  // entries (channel 2p, channel 2p+1) at inputs 2t, 2t+1, 2t+8, 2t+9
    const uint32_t l0 = lds32(lut_addr<F, n0 + 0>(w, lanebase)), l1 = lds32(lut_addr<F, n0 + 1>(w, lanebase));
    const uint32_t l2 = lds32(lut_addr<F, n0 + 2>(w, lanebase)), l3 = lds32(lut_addr<F, n0 + 3>(w, lanebase));
    r[0] = __byte_perm(l0, l1, 0x5410);
    r[1] = __byte_perm(l2, l3, 0x5410);
    r[2] = __byte_perm(l0, l1, 0x7632);
    r[3] = __byte_perm(l2, l3, 0x7632);
  } else {
    constexpr int n0 = (S * 4 + M) * 8;  // index (e, c) at n0 + 2e + c: channel 2p + c at input e
    uint32_t l[8];
    l[0] = lds32(lut_addr<F, n0 + 0>(w, lanebase));
    l[1] = lds32(lut_addr<F, n0 + 1>(w, lanebase));
    l[2] = lds32(lut_addr<F, n0 + 2>(w, lanebase));
    l[3] = lds32(lut_addr<F, n0 + 3>(w, lanebase));
    l[4] = lds32(lut_addr<F, n0 + 4>(w, lanebase));
    l[5] = lds32(lut_addr<F, n0 + 5>(w, lanebase));
    l[6] = lds32(lut_addr<F, n0 + 6>(w, lanebase));
    l[7] = lds32(lut_addr<F, n0 + 7>(w, lanebase));
    r[0] = __byte_perm(l[0], l[2], 0x5410);
    r[1] = __byte_perm(l[4], l[6], 0x5410);
    r[2] = __byte_perm(l[1], l[3], 0x5410);
    r[3] = __byte_perm(l[5], l[7], 0x5410);
  }
}

// 16-channel tile M of a decoded A tile, 16-input steps [s_lo, s_lo + n) of the K step,
// into the 16 TMEM lanes at taddr (the tile's first column): all lookups first, then the
// stores (8 columns per step).
template <int F, int M>
__device__ __forceinline__ void tmem_store_m(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase, int s_lo, int n,
                                             uint32_t taddr) {
  uint32_t r0[4], r1[4], r2[4], r3[4];
  if (s_lo <= 0 && 0 < s_lo + n) tmem_frag<F, 0, M>(w, lanebase, r0);
  if (s_lo <= 1 && 1 < s_lo + n) tmem_frag<F, 1, M>(w, lanebase, r1);
  if (s_lo <= 2 && 2 < s_lo + n) tmem_frag<F, 2, M>(w, lanebase, r2);
  if (s_lo <= 3 && 3 < s_lo + n) tmem_frag<F, 3, M>(w, lanebase, r3);
  if (s_lo <= 0 && 0 < s_lo + n) tmem_st16x256(taddr + 0u, r0);
  if (s_lo <= 1 && 1 < s_lo + n) tmem_st16x256(taddr + 8u, r1);
  if (s_lo <= 2 && 2 < s_lo + n) tmem_st16x256(taddr + 16u, r2);
  if (s_lo <= 3 && 3 < s_lo + n) tmem_st16x256(taddr + 24u, r3);
}

template <int F>
__device__ __forceinline__ void tmem_store(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase, int M, int s_lo,
                                           int n, uint32_t taddr) {
  switch (M) {
    case 0: tmem_store_m<F, 0>(w, lanebase, s_lo, n, taddr); break;
    case 1: tmem_store_m<F, 1>(w, lanebase, s_lo, n, taddr); break;
    case 2: tmem_store_m<F, 2>(w, lanebase, s_lo, n, taddr); break;
    default: tmem_store_m<F, 3>(w, lanebase, s_lo, n, taddr); break;
  }
}

// Shared-memory plan of one CTA for tiles of N rows: G = 256 / N output tiles per K step
// share one activation tile, so every step carries 128 x 256 x 64 multiply-adds whatever N.
template <int N, int F>
struct PfSmem {
  static constexpr int kG = kTileCols / N;
  static constexpr int kBTile = N * 64 * 2;
  static constexpr int kSu = FmtSizes<F>::kSuBytes;
  static constexpr int kIdxBytes = 2 * kG * kSu;  // index strings of the step's 2G super-units
  static constexpr int kLoadBytes = kBTile + kIdxBytes;
  // decoded A stages in tensor memory, after the kTileCols accumulator columns
  static constexpr int kAStages = kG >= 4 ? 2 : 3;
  static_assert(kTileCols + kAStages * kG * kACols <= kTmemCols && kAStages <= kMaxAStages, "tensor memory");
  static_assert(kBTile % 1024 == 0 && kIdxBytes % 1024 == 0, "1 KB aligned tiles");
  // codebook tables (with alignment slack), the SwiGLU exchange, alignment slack of the
  // stage area; and room for the kernel's static shared memory
  static constexpr int kTabBytes = 2 * (int)PfTab<F>::kStride;
  static constexpr int kXch = 64 * 16 * 4;
  static constexpr int kFixed = (int)PfTab<F>::kStride + kTabBytes + kXch + 1024;
  static constexpr int kStaticRoom = 6 * 1024;  // barriers and the split-group lists
  static constexpr int kFit = (227 * 1024 - kStaticRoom - kFixed) / kLoadBytes;
  static constexpr int kLoadStages = kFit > kMaxStages ? kMaxStages : kFit;
  static_assert(kLoadStages >= 2, "stage counts");
  // offsets from the kStride aligned base: tables first, then the SwiGLU exchange, the B
  // tiles (1 KB aligned) and the index strings
  static constexpr int kXchOffset = kTabBytes;
  static constexpr int kBOffset = kTabBytes + kXch;  // a multiple of 1 KB
  static constexpr int kIOffset = kBOffset + kLoadStages * kBTile;
  static constexpr int kTotal = (int)PfTab<F>::kStride + kIOffset + kLoadStages * kIdxBytes;
  static_assert(kTotal + kStaticRoom <= 227 * 1024, "shared memory per CTA");
};

// This CTA's share of the (tile group x row tile, K step) space: units [begin(c), begin(c + 1)).
__host__ __device__ __forceinline__ long long range_begin(int c, long long work, int grid) {
  return work * c / grid;
}
// CTA owning unit u (the largest c with range_begin(c) <= u).
__device__ __forceinline__ int cta_of_unit(long long u, long long work, int grid) {
  return (int)(((u + 1) * grid - 1) / work);
}

// One segment of a CTA's range: K steps [k0, k1) of tile-group row tile q.
struct Seg {
  int q, k0, k1;
};
__device__ __forceinline__ Seg seg_at(long long s, long long s1, int n_kg) {
  Seg g;
  g.q = (int)(s / n_kg);
  g.k0 = (int)(s - (long long)g.q * n_kg);
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
static_assert(2 * PfSmem<64, VQ3_FORMAT_2X16>::kTotal > 228 * 1024 && 2 * PfSmem<128, VQ3_FORMAT_2X16>::kTotal > 228 * 1024,
              "one prefill CTA per SM");

// Channel of a tile held by TMEM lane l (0 .. 127): lanes 0-63 the tile's first
// super-unit, 64-127 its second, each as 4 tiles of 16 channels in which lane g < 8 holds
// channel 2g and lane g + 8 channel 2g + 1 (tmem_frag's order).
__device__ __forceinline__ int tile_channel(int l) {
  const int m = (l & 63) >> 4, r = l & 15;
  return (l & 64) + 16 * m + (r < 8 ? 2 * r : 2 * (r - 8) + 1);
}

// Geometry of one launch, the same in every role.
struct PfGeo {
  int n_kg, n_rt, m_tiles, n_mg;
  long long work;
  __device__ PfGeo(const PrefillArgs& a, int N) {
    n_kg = a.d_in / 64;
    n_rt = (a.rows + N - 1) / N;
    n_mg = a.d_out / 64;
    m_tiles = a.swiglu ? n_mg : (n_mg + 1) / 2;
    work = a.work;
  }
};

template <int N, int F>
__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(const __grid_constant__ PrefillArgs a,
                                                                     const __grid_constant__ CUtensorMap xmap,
                                                                     const __grid_constant__ CUtensorMap imap0,
                                                                     const __grid_constant__ CUtensorMap imap1) {
  extern __shared__ __align__(16) unsigned char dsm[];
  using PS = PfSmem<N, F>;
  constexpr int G = PS::kG;
  constexpr int kSL = PS::kLoadStages;
  constexpr int kAS = PS::kAStages;
  __shared__ __align__(8) unsigned long long s_bars[2 * kMaxStages + 2 * kMaxAStages + 3];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;  // set once a wait of this CTA gave up or saw status 3
  // tile groups split between CTAs, summed after the grid barrier: [0, kMaxGrid) per CTA
  // boundary, then the list of split groups; per listed group its first and last CTA and
  // the first CTA's part slot
  __shared__ int s_split[2 * kMaxGrid];
  __shared__ int s_split_ca[kMaxGrid], s_split_cb[kMaxGrid], s_split_slot[kMaxGrid];
  __shared__ int s_nsplit;
  volatile int* abort = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = smem_u32(dsm);
  const uint32_t tabs = (raw + PfTab<F>::kStride - 1) & ~(PfTab<F>::kStride - 1);  // tables; the rest follows
  float* xch = reinterpret_cast<float*>(dsm + (tabs - raw) + PS::kXchOffset);  // up values for SwiGLU
  const uint32_t bar0 = smem_u32(s_bars);
  auto load_full = [&](int s) { return bar0 + 8u * s; };                       // B and indices landed
  auto load_empty = [&](int s) { return bar0 + 8u * (kSL + s); };              // B and indices consumed
  auto a_full = [&](int s) { return bar0 + 8u * (2 * kSL + s); };         // A decoded into tensor memory
  auto a_empty = [&](int s) { return bar0 + 8u * (2 * kSL + kAS + s); };  // A consumed
  const uint32_t acc_full = bar0 + 8u * (2 * kSL + 2 * kAS);       // the accumulators hold a finished segment
  const uint32_t acc_empty = bar0 + 8u * (2 * kSL + 2 * kAS + 1);  // the epilogue has read them
  const uint32_t mma_drain = bar0 + 8u * (2 * kSL + 2 * kAS + 2);  // every MMA issued has completed
  auto b_tile = [&](int s) { return tabs + (uint32_t)(PS::kBOffset + s * PS::kBTile); };
  auto i_tile = [&](int s) { return tabs + (uint32_t)(PS::kIOffset + s * PS::kIdxBytes); };

  const PfGeo geo(a, N);
  const int n_kg = geo.n_kg;
  const long long s0 = range_begin(blockIdx.x, a.work, gridDim.x);
  const long long s1 = range_begin(blockIdx.x + 1, a.work, gridDim.x);
  const int q_first = (int)(s0 / n_kg);  // the tile group row tile of this CTA's first unit
  // tile g of tile group tg exists; super-unit j (of 2G) of the step holds indices
  auto tile_live = [&](int tg, int g) { return tg * G + g < geo.m_tiles; };
  auto su_live = [&](int tg, int j) {
    return a.swiglu ? tile_live(tg, j % G) : 2 * tg * G + j < geo.n_mg;
  };

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
    for (int s = 0; s < kAS; ++s) {
      mbar_init(a_full(s), kDecWarps * 32);
      mbar_init(a_empty(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiThreads);
    mbar_init(mma_drain, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"((uint32_t)kTmemCols)
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
      constexpr uint32_t kTx = (uint32_t)PS::kLoadBytes;
      constexpr int kSuU4 = FmtSizes<F>::kSuUint4;
      int it = 0;
      for (long long s = s0; s < s1 && !*abort;) {
        const Seg g = seg_at(s, s1, n_kg);
        const int tg = g.q / geo.n_rt, row0 = (g.q - tg * geo.n_rt) * N;
        // the step's super-units: gate tiles then up tiles of the group (SwiGLU), or the
        // 2G channel groups of the group's tiles; an index box past the last channel group
        // reads as zeros
        const int mg0 = a.swiglu ? tg * G : 2 * tg * G;
        for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
          const int ls = it % kSL;
          if (it >= kSL) mbar_wait(load_empty(ls), (uint32_t)((it / kSL - 1) & 1), a.status, abort);
          if (*abort) break;  // a wait gave up: no further copies
          // L2 prefetch of the index strings, one span of kPrefetchSpan steps ahead (two at the
          // segment's start)
          const int j = kk - g.k0;
          if (j % kPrefetchSpan == 0) {
            const int p0 = j == 0 ? kk : kk + kPrefetchSpan;
            const int p1 = kk + 2 * kPrefetchSpan < g.k1 ? kk + 2 * kPrefetchSpan : g.k1;
            if (p1 > p0) {
              for (int su = 0; su < 2 * G; ++su) {
                if (!su_live(tg, su)) continue;
                const uint4* base = (a.swiglu && su >= G) ? a.packed1 : a.packed0;
                const int mg = a.swiglu ? mg0 + su % G : mg0 + su;
                prefetch_l2(base + ((size_t)mg * n_kg + p0) * kSuU4, (uint32_t)((p1 - p0) * PS::kSu));
              }
            }
          }
          mbar_expect_tx(load_full(ls), kTx);
          // activation tile: N rows x 64 inputs in the 128-byte swizzle layout (rows past the
          // last are filled with zeros); then the index strings of the step's super-units
          tma_load_2d(b_tile(ls), &xmap, kk * 64, row0, load_full(ls));
          tma_load_4d(i_tile(ls), &imap0, 0, 0, kk, mg0, load_full(ls));
          if (a.swiglu) tma_load_4d(i_tile(ls) + (uint32_t)(G * PS::kSu), &imap1, 0, 0, kk, mg0, load_full(ls));
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
    // Warp w writes tensor-memory lanes 32 (w % 4) .. +31 of the step's A tiles. Lanes 0-63 of
    // a tile hold its first super-unit (SwiGLU: the gate channels; otherwise the even channel
    // group), lanes 64-127 the second (up; odd), each as 4 tiles of 16 channels in the order of
    // tmem_frag; so quarter q holds 16-channel tiles 2 (q % 2) and 2 (q % 2) + 1 of super-unit
    // q / 2. The two warps of a quarter take alternate tiles of the step (with one tile per
    // step, two of its four 16-input steps each).
    const int qw = warp & 3, sub = (warp - kDecWarp0) >> 2;  // sub: 0 .. 3 within the quarter
    const int half = qw & 1, second = qw >> 1;
    constexpr int kTilesPerWarp = 1;
    constexpr int kSteps16 = G;  // 16-input steps of its tile per warp: G tiles x 4 steps over 4 warps
    const int s_lo = G >= 4 ? 0 : (G == 2 ? (sub & 1) * 2 : sub);
    // the table base (kStride aligned: its low bits are free for the entry and the lane)
    const uint32_t lanebase = (tabs + ((a.swiglu && second) ? PfTab<F>::kStride : 0u)) | (uint32_t)(lane * 4);
    const uint32_t lane_q = (uint32_t)(32 * qw) << 16;
    constexpr int kW = Fmt<F>::kWords / 4;  // words per 16-input step
    int it = 0;
    for (long long s = s0; s < s1;) {
      const Seg g = seg_at(s, s1, n_kg);
      const int tg = g.q / geo.n_rt;
      for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
        const int ls = it % kSL, as = it % kAS;
        if (it >= kAS) mbar_wait(a_empty(as), (uint32_t)((it / kAS - 1) & 1), a.status, abort);
        tc_fence_after();  // the MMAs that read this A stage are complete: it may be rewritten
        mbar_wait(load_full(ls), (uint32_t)((it / kSL) & 1), a.status, abort);
        // one decision per warp: tcgen05.st is warp-collective
        const bool go = __shfl_sync(0xffffffffu, *abort, 0) == 0;
        if (go) {
#pragma unroll 1
          for (int ti = 0; ti < kTilesPerWarp; ++ti) {
            const int t = G >= 4 ? sub : (G == 2 ? sub >> 1 : 0);
            (void)ti;
            const int su = a.swiglu ? (second ? G + t : t) : 2 * t + second;  // in the load stage
            if (!su_live(tg, su)) continue;
            uint32_t w[Fmt<F>::kWords] = {};
            const uint32_t is = i_tile(ls) + (uint32_t)(su * PS::kSu);
#pragma unroll
            for (int q = 0; q < FmtSizes<F>::kChunks; ++q) {
              if (4 * q > kW * (s_lo + kSteps16) || 4 * q + 3 < kW * s_lo) continue;
              const uint32_t o = is + (uint32_t)((q * 32 + lane) * 16);
              uint32_t v0, v1, v2, v3;
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3) : "r"(o));
              w[4 * q + 0] = v0;
              w[4 * q + 1] = v1;
              w[4 * q + 2] = v2;
              w[4 * q + 3] = v3;
            }
            const uint32_t acol = tmem + lane_q + (uint32_t)(kTileCols + (as * G + t) * kACols);
            tmem_store<F>(w, lanebase, 2 * half, s_lo, kSteps16, acol);
            tmem_store<F>(w, lanebase, 2 * half + 1, s_lo, kSteps16, acol + (16u << 16));
          }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();  // the tensor-memory writes, before the MMA thread's barrier wait
        mbar_arrive(a_full(as));
      }
      s += g.k1 - g.k0;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // A (the decoded weights) from tensor memory, B (the activations) from shared memory;
    // the accumulators of tile t at columns t N .. t N + N - 1, one segment at a time. The
    // whole warp runs the loop (warp-uniform operands); one elected lane issues.
    {
      const uint32_t idesc = idesc_f16(kTileM, N);
      int it = 0, sq = 0;
      for (long long s = s0; s < s1; ++sq) {
        const Seg g = seg_at(s, s1, n_kg);
        const int tg = g.q / geo.n_rt;
        if (sq >= 1) mbar_wait(acc_empty, (uint32_t)((sq - 1) & 1), a.status, abort);
        tc_fence_after();
        for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
          const int ls = it % kSL, as = it % kAS;
          mbar_wait(load_full(ls), (uint32_t)((it / kSL) & 1), a.status, abort);
          mbar_wait(a_full(as), (uint32_t)((it / kAS) & 1), a.status, abort);
          // a wait gave up: no further MMAs (the consumers return at once); one decision per warp
          if (__shfl_sync(0xffffffffu, *abort, 0)) continue;
          tc_fence_after();
          // one descriptor per step: K = 16 moves 8 columns along the A tile and 32 bytes (2
          // descriptor units) along the swizzled B rows
          const uint64_t bd = smem_desc_sw128(b_tile(ls));
          const uint32_t at0 = tmem + (uint32_t)(kTileCols + as * G * kACols);
          const uint32_t first = kk > g.k0 ? 1u : 0u;
#pragma unroll
          for (int t = 0; t < G; ++t) {
            if (!tile_live(tg, t)) continue;
            mma_ts_kstep(tmem + (uint32_t)(t * N), at0 + (uint32_t)(t * kACols), bd, idesc, first);
          }
          mma_commit_elect(load_empty(ls));  // both complete when this step's MMAs have read their operands
          mma_commit_elect(a_empty(as));
        }
        mma_commit_elect(acc_full);
        s += g.k1 - g.k0;
      }
      // every MMA issued has completed before the tensor memory is freed (at once unless a
      // wait gave up and the epilogue stopped waiting for the accumulators)
      mma_commit_elect(mma_drain);
      mbar_drain(mma_drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // TMEM lanes 32*(warp % 4) .. +31 = tile rows = output channels of the tile. A segment
    // that covers its tile group's whole K range is finished here; a part of a tile group
    // split between CTAs goes to this CTA's part slot (0: its first segment, 1: its last)
    // and is finished after the grid barrier below.
    // TMEM lane `row` holds channel tile_channel(row) of the tile (the decoders' order)
    const int row = (warp & 3) * 32 + lane;
    const int chan = tile_channel(row);
    int sq = 0;
    for (long long s = s0; s < s1; ++sq) {
      const Seg g = seg_at(s, s1, n_kg);
      const int tg = g.q / geo.n_rt, row0 = (g.q - tg * geo.n_rt) * N;
      const int cols = a.rows - row0 < N ? a.rows - row0 : N;  // valid rows of this tile
      mbar_wait(acc_full, (uint32_t)(sq & 1), a.status, abort);
      tc_fence_after();
      const bool whole = g.k0 == 0 && g.k1 == n_kg;
      for (int t = 0; t < G; ++t) {
        // tile_live is uniform over the epilogue's warps (the bar.sync below needs all 128 threads);
        // after an abort the loop still runs, on whatever the accumulators hold
        if (!tile_live(tg, t)) continue;
        const int mt = tg * G + t;
        const uint32_t taddr = tmem + (uint32_t)(t * N) + ((uint32_t)((warp & 3) * 32) << 16);
        if (!whole) {
          const int slot = g.q == q_first ? 0 : 1;
          float* part = a.part + (((size_t)blockIdx.x * 2 + slot) * G + t) * (size_t)kTileM * N;
#pragma unroll 1
          for (int c0 = 0; c0 < cols; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + (uint32_t)c0, r);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (VQ3_IN((size_t)(part - a.part) + (size_t)(c0 + j) * kTileM + row,
                         (size_t)gridDim.x * 2 * G * kTileM * N, 1))
                __stcg(part + (size_t)(c0 + j) * kTileM + row, __uint_as_float(r[j]));
          }
        } else if (!a.swiglu) {
          const int ch = mt * kTileM + chan;
          const bool live = ch < a.d_out;
          const float sc = live ? __half2float(__ushort_as_half(a.scale0[ch])) : 0.f;
#pragma unroll 1
          for (int c0 = 0; c0 < cols; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + (uint32_t)c0, r);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float v = __uint_as_float(r[j]) * sc;
              const int rr = row0 + c0 + j;
              if (live && c0 + j < cols && VQ3_IN((size_t)rr * a.d_out + ch, (size_t)a.rows * a.d_out, 2)) {
                if (a.lr_y) v += __ldg(a.lr_y + (size_t)rr * a.d_out + ch);  // low-rank correction
                a.out16[(size_t)rr * a.d_out + ch] = __half_as_ushort(__float2half_rn(v));
              }
            }
          }
        } else {
          // lanes 0-63: gate channels, lanes 64-127: the up channels of the same 64 (lane l + 64
          // holds the channel of lane l)
          const int jch = mt * 64 + (chan & 63);
          const bool up = row >= 64;
          const float sc = __half2float(__ushort_as_half(up ? a.scale1[jch] : a.scale0[jch]));
#pragma unroll 1
          for (int c0 = 0; c0 < cols; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + (uint32_t)c0, r);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (up) {
#pragma unroll
              for (int j = 0; j < 16; ++j) xch[j * 64 + (row - 64)] = sc * __uint_as_float(r[j]);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (!up) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float hv = silu_f(sc * __uint_as_float(r[j])) * xch[j * 64 + row];
                if (c0 + j < cols && VQ3_IN((size_t)(row0 + c0 + j) * a.d_out + jch, (size_t)a.rows * a.d_out, 3))
                  __stcg(a.out32 + (size_t)(row0 + c0 + j) * a.d_out + jch, hv);
              }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty);
      s += g.k1 - g.k0;
    }
  }

  // ------------------------------------------------------------ tile groups split between CTAs
  // Every CTA has written its parts; after a grid-wide barrier all CTAs sum them, each a
  // share of (tile group, tile, 16-row block) chunks, the parts of a chunk in CTA (= K) order.
  tc_fence_before();
  __syncthreads();
  unsigned* bar_arrive = a.flags;
  unsigned* bar_leave = a.flags + 1;
  if (tid == 0 && !*abort) {
    __threadfence();
    atomicAdd(bar_arrive, 1u);
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned spin = 1; ld_acquire_u32(bar_arrive) < gridDim.x; ++spin) {
      __nanosleep(64);
      if ((spin & 255u) == 0u) {
        if (*(volatile int*)a.status == 3 || globaltimer_ns() - t0 > kWaitNs) {
          atomicExch(a.status, 3);
          *abort = 1;
          break;
        }
      }
    }
  }
  __syncthreads();
  // Split tile groups are those holding a CTA boundary inside their K range: thread c - 1
  // looks at the boundary of CTA c, then thread 0 keeps each split group once, with its
  // first and last CTA and the first CTA's slot (0 if its range starts in the group).
  if (!*abort) {
    for (int c = tid + 1; c < (int)gridDim.x; c += kPThreads) {
      const long long u = range_begin(c, a.work, gridDim.x);
      s_split[c] = (u % n_kg) ? (int)(u / n_kg) : -1;
    }
    __syncthreads();
    if (tid == 0) {
      int n = 0, prev = -1;
      for (int c = 1; c < (int)gridDim.x; ++c) {
        const int q = s_split[c];
        if (q < 0 || q == prev) continue;
        prev = q;
        s_split[kMaxGrid + n] = q;
        ++n;
      }
      s_nsplit = n;
    }
    __syncthreads();
    // entries kMaxGrid .. kMaxGrid + n: the split groups; their CTA ranges follow
    const int n_split = s_nsplit;
    for (int i = tid; i < n_split; i += kPThreads) {
      const int q = s_split[kMaxGrid + i];
      const long long u0 = (long long)q * n_kg;
      const int ca = cta_of_unit(u0, a.work, gridDim.x);
      s_split_ca[i] = ca;
      s_split_cb[i] = cta_of_unit(u0 + n_kg - 1, a.work, gridDim.x);
      s_split_slot[i] = range_begin(ca, a.work, gridDim.x) / n_kg == q ? 0 : 1;
    }
    __syncthreads();
    const int n_c16 = N / 16;
    const size_t tile_floats = (size_t)kTileM * N;
    const size_t cta_floats = 2 * (size_t)G * tile_floats;  // a CTA's two part slots
    const long long n_chunks = (long long)n_split * G * n_c16;
    // this CTA's chunks are c = blockIdx.x + k grid; their items (a float4 of 4 lanes of one
    // accumulator row, or for SwiGLU a gate float4 with its up float4) run as one flat loop
    // over all threads
    const int ipc = a.swiglu ? 16 * 16 : kTileM / 4 * 16;  // items per chunk
    const long long my_chunks = n_chunks > blockIdx.x ? (n_chunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const size_t stride4 = cta_floats / 4;
    auto add4 = [](float4& v, const float4 x) {
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    };
    for (long long item = tid; item < my_chunks * ipc; item += kPThreads) {
      const long long c = blockIdx.x + (item / ipc) * gridDim.x;
      const int e = (int)(item % ipc);
      const int i = (int)(c / (G * n_c16)), t = (int)(c / n_c16 % G), c16 = (int)(c % n_c16);
      const int q = s_split[kMaxGrid + i];
      const int tg = q / geo.n_rt, row0 = (q - tg * geo.n_rt) * N;
      const int cols = a.rows - row0 < N ? a.rows - row0 : N;
      if (!tile_live(tg, t)) continue;
      const int mt = tg * G + t;
      const int ca = s_split_ca[i], np = s_split_cb[i] - ca + 1;
      // the parts in CTA (= K) order: CTA ca's in its slot, the later CTAs' in slot 0; a part
      // is [16 rows of the tile][128 lanes] FP32 here, read four lanes at a time
      const float4* p0 = reinterpret_cast<const float4*>(a.part + (size_t)ca * cta_floats +
                                                         (size_t)s_split_slot[i] * G * tile_floats +
                                                         (size_t)t * tile_floats + (size_t)c16 * 16 * kTileM);
      const float4* p1 = reinterpret_cast<const float4*>(a.part + (size_t)(ca + 1) * cta_floats +
                                                         (size_t)t * tile_floats + (size_t)c16 * 16 * kTileM);
      auto sum_parts = [&](int off4) {
        if (!VQ3_IN((size_t)(p0 - reinterpret_cast<const float4*>(a.part)) + off4, (size_t)gridDim.x * stride4, 4) ||
            (np > 1 && !VQ3_IN((size_t)(p1 - reinterpret_cast<const float4*>(a.part)) + (size_t)(np - 2) * stride4 + off4,
                                (size_t)gridDim.x * stride4, 5)))
          return make_float4(0.f, 0.f, 0.f, 0.f);
        float4 v = __ldcg(p0 + off4);
        int p = 0;
        for (; p + 8 <= np - 1; p += 8) {
          float4 x[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) x[k] = __ldcg(p1 + (size_t)(p + k) * stride4 + off4);
#pragma unroll
          for (int k = 0; k < 8; ++k) add4(v, x[k]);
        }
        for (; p < np - 1; ++p) add4(v, __ldcg(p1 + (size_t)p * stride4 + off4));
        return v;
      };
      if (!a.swiglu) {
        const int f = e % (kTileM / 4), j = e / (kTileM / 4);  // lanes 4f .. 4f+3, row j of the chunk
        const int rr = row0 + c16 * 16 + j;
        if (c16 * 16 + j >= cols) continue;
        const float4 v = sum_parts(j * (kTileM / 4) + f);
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ch = mt * kTileM + tile_channel(4 * f + k);
          if (ch >= a.d_out || !VQ3_IN((size_t)rr * a.d_out + ch, (size_t)a.rows * a.d_out, 6)) continue;
          float o = vv[k] * __half2float(__ushort_as_half(a.scale0[ch]));
          if (a.lr_y) o += __ldg(a.lr_y + (size_t)rr * a.d_out + ch);
          a.out16[(size_t)rr * a.d_out + ch] = __half_as_ushort(__float2half_rn(o));
        }
      } else {
        const int f = e % 16, j = e / 16;  // gate lanes 4f .. 4f+3 and the up lanes 64 on
        const int rr = row0 + c16 * 16 + j;
        if (c16 * 16 + j >= cols) continue;
        const float4 gv = sum_parts(j * (kTileM / 4) + f), uv = sum_parts(j * (kTileM / 4) + 16 + f);
        const float g4[4] = {gv.x, gv.y, gv.z, gv.w}, u4[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int jch = mt * 64 + tile_channel(4 * f + k);
          const float sg = __half2float(__ushort_as_half(a.scale0[jch]));
          const float su2 = __half2float(__ushort_as_half(a.scale1[jch]));
          if (VQ3_IN((size_t)rr * a.d_out + jch, (size_t)a.rows * a.d_out, 7))
            __stcg(a.out32 + (size_t)rr * a.d_out + jch, silu_f(sg * g4[k]) * (su2 * u4[k]));
        }
      }
    }
  }
  // the last CTA out clears the barrier words for the next launch
  __syncthreads();
  if (tid == 0) {
    const unsigned old = atomicAdd(bar_leave, 1u);
    if (old + 1 == gridDim.x) {
      *(volatile unsigned*)bar_arrive = 0u;
      *(volatile unsigned*)bar_leave = 0u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)kTmemCols)
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

// The GPU-layout indices of one matrix as a 4D byte tensor [channel group][K step][SU row]
// [256 bytes] (an SU of su_bytes = rows x 256 bytes), read `groups` channel groups of one
// K step at a time: the step's super-units land back to back. Boxes past the last channel
// group read as zeros.
cudaError_t index_map(const void* packed, int d_in, int d_out, int su_bytes, int groups, CUtensorMap* map) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const int n_kg = d_in / 64, n_mg = d_out / 64, su_rows = su_bytes / 256;
  const cuuint64_t dims[4] = {256, (cuuint64_t)su_rows, (cuuint64_t)n_kg, (cuuint64_t)n_mg};
  const cuuint64_t strides[3] = {256, (cuuint64_t)su_bytes, (cuuint64_t)n_kg * su_bytes};
  const cuuint32_t box[4] = {256, (cuuint32_t)su_rows, 1, (cuuint32_t)groups};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(packed), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int N, int F>
cudaError_t launch_n(PrefillArgs a, cudaStream_t st) {
  using PS = PfSmem<N, F>;
  const int smem = PS::kTotal;
  cudaError_t e = cudaFuncSetAttribute(prefill_gemm_kernel<N, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap xmap, imap0, imap1;
  if ((e = activation_map(a, N, &xmap)) != cudaSuccess) return e;
  const int groups = a.swiglu ? PS::kG : 2 * PS::kG;
  if ((e = index_map(a.packed0, a.d_in, a.d_out, PS::kSu, groups, &imap0)) != cudaSuccess) return e;
  if ((e = index_map(a.swiglu ? a.packed1 : a.packed0, a.d_in, a.d_out, PS::kSu, groups, &imap1)) != cudaSuccess)
    return e;
  a.work = prefill_work(a.rows, a.d_in, a.d_out, a.swiglu);
  const int grid = prefill_grid(a.rows, a.d_in, a.d_out, a.swiglu);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: the grid barrier before the split sums
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<N, F>, a, xmap, imap0, imap1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int prefill_tile_rows(int rows) { return rows > 64 ? 128 : 64; }  // this kernel serves up to 128 rows

long long prefill_work(int rows, int d_in, int d_out, int swiglu) {
  const long long m_tiles = swiglu ? d_out / 64 : (d_out / 64 + 1) / 2;
  const int n = prefill_tile_rows(rows);
  const long long groups = (m_tiles + kTileCols / n - 1) / (kTileCols / n);
  return groups * ((rows + n - 1) / n) * (d_in / 64);
}

int prefill_max_grid() { return device_sm_count() < kMaxGrid ? device_sm_count() : kMaxGrid; }

int prefill_grid(int rows, int d_in, int d_out, int swiglu) {
  const long long work = prefill_work(rows, d_in, d_out, swiglu);
  const long long g = work / kMinSteps;
  const int cap = prefill_max_grid();
  return g < 1 ? 1 : (g < cap ? (int)g : cap);
}

size_t prefill_part_bytes(int rows) {
  (void)rows;  // two slots per CTA of G tiles x 128 channels x N rows = 128 x 256 FP32 whatever N
  return (size_t)prefill_max_grid() * 2 * kTileM * kTileCols * sizeof(float);
}

namespace {
template <int F>
cudaError_t launch_fmt(const PrefillArgs& a, cudaStream_t st) {
  if (a.rows > 2 * 64) return cudaErrorInvalidValue;  // wider tiles: launch_prefill_wide_gemm
  return prefill_tile_rows(a.rows) == 64 ? launch_n<64, F>(a, st) : launch_n<128, F>(a, st);
}
}  // namespace

cudaError_t launch_prefill_gemm(const PrefillArgs& a, cudaStream_t st) {
  switch (a.format) {
    case VQ3_FORMAT_2X64: return launch_fmt<VQ3_FORMAT_2X64>(a, st);
    case VQ3_FORMAT_2X16: return launch_fmt<VQ3_FORMAT_2X16>(a, st);
    case VQ3_FORMAT_LUT4: return launch_fmt<VQ3_FORMAT_LUT4>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vq3
