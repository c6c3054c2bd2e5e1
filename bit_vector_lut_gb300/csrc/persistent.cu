// The small-row-count path (T <= 32 rows per pass) of the VQ3 MLP block and of
// a single VQ3 linear layer: one persistent cooperative kernel per pass.
//
// What it computes (model card "anemll/anemll-forge-qwen3.8-27B", section
// "Release 0.2: three-bit MLP, token-mixer rotations, distilled weights": every
// MLP matrix a 2x64 vector LUT with per-channel scales, each matrix input
// multiplied online by blocked Hadamard matrices with seeded signs; SiLU as
// x*sigmoid(x) per "ANEMLL ANE LLM conversion pipeline", section "Facts"):
//   g, u = W_g R_in x, W_u R_in x      decode, split-K partial sums ("pieces")
//   h    = silu(s_g g) * (s_u u)       one task per 64 intermediate channels
//   y    = W_d R_dn h                  decode, pieces
//   out  = fp16(s_d y)                 one task per 64 output channels x 8-row tile
// A single matrix runs the first decode and the output tasks (adding its low-rank
// correction U V x' when it has factors).
//
// In a stacked layer the pre-norm residual step is folded in: either the prologue
// forms r' = fp16(x + delta) over whole rows and its RMS, or the RMS comes from the
// previous layer's partial sums of squares; the x rotation normalises on the fly,
// and the output tasks can also write r + out and that row's new partial sums.
//
// The rotations R = blockdiag(H_b diag(s)) / sqrt(b) are not separate steps: a
// decoding CTA rotates the chunks of x (or h) its column groups lie in, straight
// into its shared-memory activation stage. x is an input; h is complete per chunk
// when that chunk's SwiGLU tasks have counted themselves done.
//
// There are no grid-wide barriers. Every consumer waits only for what it reads,
// through counters in the workspace: segment groups count the CTAs that wrote
// their pieces, h chunks count finished SwiGLU tasks. Waits are bounded in time
// (on timeout the status word gets 3 and the kernel still ends). The
// cooperative launch makes all CTAs co-resident and no wait depends on work
// ordered after it in any CTA, so every wait ends. The last CTA to finish
// resets the counters to zero for the next launch.
//
// Decode: the m16n8k16 tensor-core path. A tcgen05.mma takes the same time for
// any N up to 256, so at N = 8..32 it would absorb ~5 indices per clock per SM,
// a sixth of what streaming the indices at HBM speed needs; m16n8k16 absorbs
// ~60, which leaves the decode itself (shift, mask, shared-memory lookup, byte
// permute per index) as the limit.
//   - Each CTA holds lane-private copies of the three codebooks (entry k of lane
//     L at word k*32 + L) at a 16 KB-aligned shared address, so a lookup is one
//     shift, one LOP3 and one bank-conflict-free load.
//   - Segments (64 output channels x matrix) are grouped 16 at a time, one per
//     warp; a cell is one group x one 64-input column group, and every CTA owns a
//     contiguous run of cells. Its activation stage holds the fragments of up to
//     32/NT cells' column groups (all 16 warps read them), and every warp streams
//     its own segment's index strings through a 3-deep cp.async ring.
//   - A warp's sum over its run of a segment is one piece; consumers sum a
//     segment's pieces in CTA (= K) order, so results do not depend on timing.
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
VQ3_BOUNDS_RECORD(persistent)
namespace {

constexpr int kWarps = kDecWarps;  // 16
constexpr int kThreads = kWarps * 32;
// Lane-private codebook tables: entry k of lane L at word k*32 + L; one table
// per matrix, kTabStride bytes apart, the pair of gate and up tables aligned to
// twice that so the matrix choice is an OR of the table offset.
template <int F>
struct Tab {
  static constexpr uint32_t kStride = (uint32_t)Fmt<F>::kEntries * 128u;  // 8 KB or 2 KB
  static constexpr uint32_t kAlign = 2u * kStride;
};
constexpr unsigned long long kWaitNs = 1000000000ull;  // a wait gives up after one second

// ------------------------------------------------------------------ primitives

// Not volatile: a pure function of its registers, free to schedule.
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared address of the lookup for lane index N: bits [b N, b N + b) of the
// lane's string (b = index width) moved to bits [7, 7 + b) (entry stride 32 lanes
// x 4 bytes), OR-ed with the table base, the lane's column and the matrix's
// table offset.
template <int F, int N>
__device__ __forceinline__ uint32_t lut_addr(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase) {
  constexpr int kB = Fmt<F>::kBits;
  constexpr int pos = kB * N;
  constexpr int wd = pos / 32;
  constexpr int off = pos % 32;
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

// The tables are read-only while cells are decoded: a pure load, free to reorder.
__device__ __forceinline__ uint32_t lut(uint32_t saddr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(saddr));
  return v;
}

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

__device__ __forceinline__ void lds64(uint32_t saddr, uint32_t& a, uint32_t& b) {
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "r"(saddr) : "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t saddr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(saddr) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t saddr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(saddr), "f"(v) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(saddr) : "memory");
  return v;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// 32-bit unsigned arithmetic throughout (the launcher checks cells * grid < 2^32):
// these run on the path between steps, where a 64-bit division costs microseconds.
__device__ __forceinline__ int range_begin(int cells, int grid, int b) {
  return (int)((unsigned)b * (unsigned)cells / (unsigned)grid);
}

// CTA owning cell x (largest b with range_begin(b) <= x).
__device__ __forceinline__ int cta_of(int x, int cells, int grid) {
  return (int)((((unsigned)x + 1u) * (unsigned)grid - 1u) / (unsigned)cells);
}

// The same partition with the cells of the first segment group weighted 1 + lw / 8 (lw > 0: a
// linear layer with low-rank factors, whose first-group CTAs also form z): in eighths of a cell,
// cell x ends at cost(x) = 8 x + lw min(x, n0), CTA b starts at the first cell whose cost reaches
// b T / grid (T = cost(cells)), and cta_of inverts that. lw = 0 is the partition above.
__device__ __forceinline__ unsigned wcost(int x, int n0, int lw) {
  return 8u * (unsigned)x + (unsigned)lw * (unsigned)(x < n0 ? x : n0);
}
__device__ __forceinline__ int range_begin_w(int cells, int grid, int b, int n0, int lw) {
  if (!lw) return range_begin(cells, grid, b);
  const unsigned T = wcost(cells, n0, lw);
  const unsigned target = (unsigned)b * T / (unsigned)grid;
  const unsigned w0 = (unsigned)(8 + lw), c0 = w0 * (unsigned)n0;
  if (target <= c0) return (int)((target + w0 - 1u) / w0);
  return n0 + (int)((target - c0 + 7u) / 8u);
}
__device__ __forceinline__ int cta_of_w(int x, int cells, int grid, int n0, int lw) {
  if (!lw) return cta_of(x, cells, grid);
  return (int)(((wcost(x, n0, lw) + 1u) * (unsigned)grid - 1u) / wcost(cells, n0, lw));
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}


// ------------------------------------------------------------------ counters

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Thread 0 polls until *p >= target. The counter is polled first, so a wait whose data is
// ready costs one acquire load. Otherwise the wait is bounded in time: after kWaitNs it
// sets the status word to 3 and returns; and once any wait of the launch has given up
// (status 3, checked every 64 polls) every wait returns at once.
__device__ __forceinline__ void poll_geq(const unsigned* p, unsigned target, int* status) {
  if (ld_acquire(p) >= target) return;
  if (*(volatile int*)status == 3) return;
  const unsigned long long t0 = globaltimer_ns();
  for (unsigned it = 1;; ++it) {
    __nanosleep(32);
    if (ld_acquire(p) >= target) return;
    if ((it & 63u) == 0u) {
      if (*(volatile int*)status == 3) return;
      if (globaltimer_ns() - t0 > kWaitNs) {
        atomicExch(status, 3);
        return;
      }
    }
  }
}

__device__ __forceinline__ void red_release(unsigned* p) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p) : "memory");
}

// The CTA's writes so far become visible, then *p += 1 (and *p2 += 1): the barrier orders
// every thread's writes before thread 0's release increments.
__device__ __forceinline__ void signal(unsigned* p, unsigned* p2) {
  __syncthreads();
  if (threadIdx.x == 0) {
    red_release(p);
    if (p2) red_release(p2);
  }
}

// ------------------------------------------------------------------ geometry

struct DecodeJob {
  int d_in, d_out, n_mats;
  const uint4* packed0;
  const uint4* packed1;
  const uint16_t* scales0;
  float* pieces;            // [n_seg][max_pieces][512 * NT]
  int grid, max_pieces;     // decoding CTAs (<= cells) and piece slots per segment
  uint32_t tab;             // shared address of matrix 0's table (16 KB aligned); matrix 1 at +8192
  // activation source, rotated into the stage: rows [0, rows) at src + r * src_ld
  size_t src_ld;
  int rows, block, chunk;   // valid rows; rotation block; chunk (whole blocks, columns)
  float scale;              // 1 / sqrt(block)
  int c0, c1;               // this CTA's cells [c0, c1) (set when the job is made)
  const uint32_t* signs;
  const float* inv;         // RMSNorm of the source rows: per-row 1/rms (shared memory), or null
  const uint16_t* res_delta;  // with inv: the residual delta added to the source first, or null
  const unsigned* ready;    // per chunk: complete when >= ready_target (null: ready at launch)
  unsigned ready_target;
  unsigned* group_done;     // per segment group: +1 per CTA whose pieces of the group are written
  // low-rank projection z = V x' (linear job with factors, else lr_v null): formed by the CTAs
  // of the first segment group from their stage slots, one partial per CTA in lr_z
  const uint16_t* lr_v;
  int lr_rank;
  float* lr_z;
  unsigned* lr_done;        // +1 per CTA whose partial of z is written
  int lw;                   // extra weight of a first-group cell in the CTA ranges, eighths (0: none)
  uint32_t zacc;            // shared address: per warp [NT][4][32 lanes] FP32 running sums

  __device__ int n_kg() const { return d_in / kSuInputs; }
  __device__ int n_seg() const { return (d_out / kSuChannels) * n_mats; }
  __device__ int n_grp() const { return (n_seg() + kWarps - 1) / kWarps; }
  __device__ int cells() const { return n_grp() * n_kg(); }
  // CTAs that write pieces of segment group g (slots 0 .. count-1)
  __device__ int contributors(int g) const {
    const int x0 = g * n_kg();
    return cta_of_w(x0 + n_kg() - 1, cells(), grid, n_kg(), lw) - cta_of_w(x0, cells(), grid, n_kg(), lw) + 1;
  }
  __device__ const float* seg_pieces(int sg, int piece_floats) const {
    return pieces + (size_t)sg * max_pieces * piece_floats;
  }
};

struct SmemView {
  uint32_t ring, stage, tab;  // shared addresses
  float* scratch;             // rotation scratch: 4 KB per warp
  int* flag;                  // one word for the last-CTA test
};

// Item `it` of a piece -> (row of the pass, channel within the 64-channel group).
// Piece layout: it = ((m * NT + nt) * 4 + j) * 32 + lane, the m16n8k16 accumulator order.
template <int NT>
__device__ __forceinline__ void item_pos(int it, int& row, int& ch) {
  const int L = it & 31, idx = it >> 5;
  const int j = idx & 3, mnt = idx >> 2, nt = mnt % NT, m = mnt / NT;
  ch = (8 * m + (L >> 2)) * 2 + (j >> 1);
  row = nt * 8 + 2 * (L & 3) + (j & 1);
}

// ------------------------------------------------------------------ rotation into the stage
//
// Stage layout: slot p (cell rs + p of the round, column group kg(p)) holds NT
// 1 KB row tiles; tile nt holds the B fragments of rows 8nt .. 8nt+7: the 16-byte
// chunk q = h*32 + 4g + t (row g, half h) carries columns 32h + 8i + 2t + {0, 1}
// (i = 0..3) of the column group as FP16 pairs. Chunk q is stored at position
// q ^ (p & 7), which keeps both the rotation's writes (one row, 16 column groups
// per warp instruction) and the decode's reads (512 contiguous bytes) free of
// bank conflicts.

template <int NT>
struct StageCfg {
  static constexpr int kSlots = NT == 1 ? 32 : (NT == 2 ? 16 : 8);  // column groups per round
  static constexpr int kBytes = kSlots * NT * 1024;
};

__device__ __forceinline__ uint32_t stage_chunk_addr(uint32_t stage, int p, int nt_count, int nt, int q) {
  return stage + (uint32_t)((p * nt_count + nt) * 1024 + ((q ^ (p & 7)) << 4));
}

__device__ __forceinline__ void sts128(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// (a * s, b * s) rounded to an FP16 pair; the products as scalar multiplies would round them.
__device__ __forceinline__ uint32_t pack_half2_scaled(float a, float b, unsigned long long ss) {
  unsigned long long x;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(x) : "l"(x), "l"(ss));
  float p, q;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(p), "=f"(q) : "l"(x));
  return pack_half2(p, q);
}

// Butterflies of stride S (in register index) over v[0 .. 32).
template <int S>
__device__ __forceinline__ void bfly32(float (&v)[32]) {
  if constexpr (S == 1) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float x0 = v[i], x1 = v[i + 1];
      v[i] = x0 + x1;
      v[i + 1] = x0 - x1;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; i += 2)
      if ((i & S) == 0) {
        const float x0 = v[i], x1 = v[i + S], y0 = v[i + 1], y1 = v[i + S + 1];
        v[i] = x0 + x1;
        v[i + S] = x0 - x1;
        v[i + 1] = y0 + y1;
        v[i + S + 1] = y0 - y1;
      }
  }
}

// 32 x 32 bit transpose across the warp: bit b of lane r's result is bit r of lane b's word.
__device__ __forceinline__ uint32_t warp_bit_transpose(uint32_t x, int lane) {
  constexpr uint32_t m[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int r = 0; r < 5; ++r) {
    const int sh = 16 >> r;
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, sh);
    x = (lane & sh) ? ((x & ~m[r]) | ((y >> sh) & m[r])) : ((x & m[r]) | ((y & m[r]) << sh));
  }
  return x;
}

// Butterflies of register strides 1 .. min(32, limit)/2.
__device__ __forceinline__ void fwht32(float (&v)[32], int limit) {
  if (limit > 1) bfly32<1>(v);
  if (limit > 2) bfly32<2>(v);
  if (limit > 4) bfly32<4>(v);
  if (limit > 8) bfly32<8>(v);
  if (limit > 16) bfly32<16>(v);
}

// Hadamard butterflies of strides 1 .. block/2 over buf[0 .. n) (n a multiple of block).
__device__ __forceinline__ void fwht_smem(float* buf, int n, int block) {
  for (int lh = 0; (1 << lh) < block; ++lh) {
    const int h = 1 << lh;
    for (int q = threadIdx.x; q < n / 2; q += kThreads) {
      const int i0 = ((q >> lh) << (lh + 1)) + (q & (h - 1)), i1 = i0 + h;
      const float x0 = buf[i0], x1 = buf[i1];
      buf[i0] = x0 + x1;
      buf[i1] = x0 - x1;
    }
    __syncthreads();
  }
}

__device__ __forceinline__ float load1(const uint16_t* p) { return __half2float(__ushort_as_half(__ldg(p))); }
__device__ __forceinline__ float load1(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float round16(float v) { return __half2float(__float2half_rn(v)); }

// Source element (row, col) of the stage: for a normed source the pre-norm residual step
// fp16(fp16(x + delta) * inv[row]), else the element itself.
template <typename T>
__device__ __forceinline__ float act(const DecodeJob& a, const T* src, int row, int col) {
  const size_t o = (size_t)row * a.src_ld + col;
  float v = VQ3_IN(o, (size_t)a.rows * a.src_ld, 2) ? load1(src + o) : 0.f;
  if constexpr (sizeof(T) == 2) {
    if (a.inv) {
      if (a.res_delta) v = round16(v + (VQ3_IN(o, (size_t)a.rows * a.src_ld, 3) ? load1(a.res_delta + o) : 0.f));
      v = round16(v * a.inv[row]);
    }
  }
  return v;
}

__device__ __forceinline__ bool sign_bit(const uint32_t* signs, int col) {
  return (__ldg(signs + (col >> 5)) >> (col & 31)) & 1u;
}

// The chunks that hold the round's column groups kg_s .. kg_s + len - 1 (cyclic over
// n_chunks chunks of 2^lg column groups; a chunk is a power of two, like the rotation
// block): n of them, from chunk first on, each once.
struct Window {
  int first, n, n_chunks;
  __device__ Window(int kg_s, int len, int lg, int n_chunks_) : n_chunks(n_chunks_) {
    first = kg_s >> lg;
    n = (kg_s - (first << lg) + len + (1 << lg) - 1) >> lg;
    if (n > n_chunks) n = n_chunks;
  }
  __device__ int chunk(int i) const { return first + i < n_chunks ? first + i : first + i - n_chunks; }
};

// Writes the stage slots of round [rs, rs + len): the rotated activations of each
// slot's column group, rows < a.rows (other rows are left as they are: an MMA
// column depends on its own B column only, and their outputs are never stored).
template <int NT, typename T>
__device__ __forceinline__ void stage_round(const DecodeJob& a, const T* src, int kg_s, int len, const SmemView& sv) {
  const int n_kg = a.n_kg();
  const int ckg = a.chunk / kSuInputs;
  const int lg = __ffs(ckg) - 1;  // ckg is a power of two
  const int n_chunks = n_kg >> lg;
  const float scale = a.scale;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (a.chunk == 1024) {
    // one (chunk, row) per warp: lane L holds columns L + 32 j, then 32 L + c
    float* m = sv.scratch + warp * 1024;
    unsigned long long ss;  // (scale, scale)
    asm("mov.b64 %0, {%1, %1};" : "=l"(ss) : "f"(scale));
    int item = 0;
    const Window win(kg_s, len, lg, n_chunks);
    for (int i = 0; i < win.n; ++i) {
      const int c = win.chunk(i);
      for (int row = 0; row < a.rows; ++row, ++item) {
        if ((item & (kWarps - 1)) != warp) continue;
        const T* s = src + (size_t)row * a.src_ld + c * 1024;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          v[j] = VQ3_IN((size_t)row * a.src_ld + c * 1024 + 32 * j + lane, (size_t)a.rows * a.src_ld, 5)
                     ? load1(s + 32 * j + lane) : 0.f;
        if constexpr (sizeof(T) == 2) {
          if (a.inv) {
            // pre-norm residual step: fp16(fp16(x + delta) * inv[row]), its loads after x's
            const float iv = a.inv[row];
            if (a.res_delta) {
              const uint16_t* sd = a.res_delta + (size_t)row * a.src_ld + c * 1024;
              float dl[32];
#pragma unroll
              for (int j = 0; j < 32; ++j)
                dl[j] = VQ3_IN((size_t)row * a.src_ld + c * 1024 + 32 * j + lane, (size_t)a.rows * a.src_ld, 6)
                            ? load1(sd + 32 * j + lane) : 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = round16(v[j] + dl[j]);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = round16(v[j] * iv);
          }
        }
        if (a.signs) {
          // bit j of t: the sign of column c * 1024 + 32 j + lane (one word per lane, transposed)
          const uint32_t t =
              warp_bit_transpose(VQ3_IN(c * 32 + lane, a.d_in / 32, 7) ? __ldg(a.signs + c * 32 + lane) : 0u, lane);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __int_as_float(__float_as_int(v[j]) ^ ((t << (31 - j)) & 0x80000000u));
        }
        fwht32(v, a.block >> 5);  // column strides 32 .. block/2
#pragma unroll
        for (int j = 0; j < 32; ++j) m[j * 32 + (lane ^ j)] = v[j];
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = m[lane * 32 + (k ^ lane)];
        __syncwarp();
        fwht32(v, a.block);  // column strides 1 .. min(block, 32)/2
        const int kg = c * ckg + (lane >> 1), h = lane & 1, nt = row >> 3, g = row & 7;
        for (int p = kg - kg_s < 0 ? kg - kg_s + n_kg : kg - kg_s; p < len; p += n_kg)
#pragma unroll
          for (int t = 0; t < 4; ++t)
            sts128(stage_chunk_addr(sv.stage, p, NT, nt, h * 32 + 4 * g + t),
                   pack_half2_scaled(v[2 * t], v[2 * t + 1], ss), pack_half2_scaled(v[8 + 2 * t], v[9 + 2 * t], ss),
                   pack_half2_scaled(v[16 + 2 * t], v[17 + 2 * t], ss),
                   pack_half2_scaled(v[24 + 2 * t], v[25 + 2 * t], ss));
      }
    }
    return;
  }
  // smaller chunks: CTA-wide butterflies over [8 rows][chunk] fp32 in the scratch
  float* buf = sv.scratch;
  const Window win(kg_s, len, lg, n_chunks);
  for (int i = 0; i < win.n; ++i) {
    const int c = win.chunk(i);
    for (int nt = 0; nt < NT; ++nt) {
      const int nr = a.rows - nt * 8 < 8 ? a.rows - nt * 8 : 8;
      if (nr <= 0) break;
      for (int e = threadIdx.x; e < nr * a.chunk; e += kThreads) {
        const int rr = e / a.chunk, col = c * a.chunk + e % a.chunk;
        float v = act(a, src, nt * 8 + rr, col);
        if (a.signs && VQ3_IN(col >> 5, a.d_in / 32, 4) && sign_bit(a.signs, col)) v = -v;
        buf[e] = v;
      }
      __syncthreads();
      fwht_smem(buf, nr * a.chunk, a.block);
      // one 16-byte fragment chunk per item: (row, column group of the chunk, h, t)
      for (int e = threadIdx.x; e < nr * ckg * 8; e += kThreads) {
        const int rr = e / (ckg * 8), kl = (e / 8) % ckg, h = (e / 4) & 1, t = e & 3;
        const float* r = buf + rr * a.chunk + kl * 64 + 32 * h + 2 * t;
        const int kg = c * ckg + kl;
        for (int p = kg - kg_s < 0 ? kg - kg_s + n_kg : kg - kg_s; p < len; p += n_kg)
          sts128(stage_chunk_addr(sv.stage, p, NT, nt, h * 32 + 4 * rr + t), pack_half2(r[0] * scale, r[1] * scale),
                 pack_half2(r[8] * scale, r[9] * scale), pack_half2(r[16] * scale, r[17] * scale),
                 pack_half2(r[24] * scale, r[25] * scale));
      }
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------------ low-rank projection
//
// z = V x' for a linear layer with factors (W = diag(s) C[idx] + U V on the rotated input:
// model card "anemll/anemll-forge-qwen3.8-27B", table row "Token mixers", rank-64 factors).
// The CTAs that decode the first segment group hold, between them, every column group's
// rotated activations in their stage slots once each, so they form z from those slots: per
// slot, warp w takes factor rows 16 (w >> 2) .. + 15 over k-step w & 3, one m16n8k16 per
// 8-row tile, into running sums of its own in shared memory (after the round's cells are
// decoded: the decode loop itself is the same as without factors). Where the CTA's part of
// the first group ends, the sums of the four k-step warps of each row tile are added in
// k-step order and written as the CTA's partial of z, and a counter of its own is raised.

// The factor columns of a batch of up to kLrBatch first-group slots sit in the rotation scratch
// (idle while cells are decoded): row q of V at q * kLrRow bytes, the batch's column groups one
// after another. The row stride is 4 words past a multiple of 32, so a fragment load (rows g,
// columns 2t) touches 32 distinct banks.
constexpr int kLrBatch = 7;
constexpr uint32_t kLrRow = kLrBatch * 128 + 16;

// Copies V's columns of column groups kg0 .. kg0 + n - 1 (n <= kLrBatch) into the scratch as
// 16-byte copies spread over the CTA's threads (consecutive threads take consecutive chunks of a
// row), committed by every thread as one copy group.
__device__ __forceinline__ void lr_copy(const DecodeJob& a, const SmemView& sv, int kg0, int n) {
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(sv.scratch));
  const int per_row = n * (kSuInputs / 8);  // 16-byte chunks of a row
  for (int i = threadIdx.x; i < a.lr_rank * per_row; i += kThreads) {
    const int q = i / per_row, k = i - q * per_row;
    if (VQ3_IN((size_t)q * a.d_in + (size_t)kg0 * kSuInputs + (size_t)k * 8, (size_t)a.lr_rank * a.d_in, 20))
      cp_async16(base + (uint32_t)q * kLrRow + (uint32_t)k * 16u,
                 a.lr_v + (size_t)q * a.d_in + (size_t)kg0 * kSuInputs + (size_t)k * 8);
  }
  cp_async_commit();
}

// Warp's share over the batch's slots: slot p of the round (column group kg0 + p) is column
// block p - b0 of the copied factor rows. Within a k-step the stage holds the inputs in natural
// order (b0: columns 2t, 2t+1; b1: 2t+8, 2t+9), as the copied rows do; rows past the rank are zero.
template <int NT>
__device__ __forceinline__ void lowrank_slots(const DecodeJob& a, const SmemView& sv, int b0, int n) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = warp & 3, t = lane & 3;
  const int qlo = 16 * (warp >> 2) + (lane >> 2), qhi = qlo + 8;
  const bool lo = qlo < a.lr_rank, hi = qhi < a.lr_rank;
  const uint32_t vs = static_cast<uint32_t>(__cvta_generic_to_shared(sv.scratch)) + (uint32_t)(16 * s + 2 * t) * 2u;
  const uint32_t vlo = vs + (uint32_t)qlo * kLrRow, vhi = vs + (uint32_t)qhi * kLrRow;
  const uint32_t zw = a.zacc + (uint32_t)(warp * NT * 128 + lane) * 4u;
  float z[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 4; ++j) z[nt][j] = lds_f32(zw + (uint32_t)((nt * 4 + j) * 128));
#pragma unroll
  for (int i = 0; i < kLrBatch; ++i) {
    if (i >= n) break;
    const uint32_t c = (uint32_t)i * 128u;
    uint32_t av[4];
    av[0] = lo ? lds32(vlo + c) : 0u;        // row g:   columns 2t, 2t+1
    av[1] = hi ? lds32(vhi + c) : 0u;        // row g+8
    av[2] = lo ? lds32(vlo + c + 16u) : 0u;  // row g:   columns 2t+8, 2t+9
    av[3] = hi ? lds32(vhi + c + 16u) : 0u;  // row g+8
    const int p = b0 + i;
    const uint32_t xb = sv.stage + (uint32_t)(p * NT * 1024) +
                        (uint32_t)((s >> 1) * 32 + (lane ^ (p & 7))) * 16u + 8u * (uint32_t)(s & 1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint32_t x0, x1;
      lds64(xb + (uint32_t)(nt * 1024), x0, x1);
      mma16816(z[nt], av, x0, x1);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 4; ++j) sts_f32(zw + (uint32_t)((nt * 4 + j) * 128), z[nt][j]);
}

// z's share of a round's first-group slots [0, n0) (column groups kg0 ..), one batch of factor
// columns at a time. Called after the round's first cell: the first batch's copy group was
// committed before the round's cells, so all but the one cell copy group committed since it
// have to be complete; a later batch waits for every group (the cells' copies in flight too).
template <int NT>
__device__ __forceinline__ void lr_round(const DecodeJob& a, const SmemView& sv, int kg0, int n0) {
  for (int b0 = 0; b0 < n0; b0 += kLrBatch) {
    const int nb = min(kLrBatch, n0 - b0);
    if (b0) {
      __syncthreads();  // the previous batch's reads of the scratch are done
      lr_copy(a, sv, kg0 + b0, nb);
      cp_async_wait<0>();
    } else {
      cp_async_wait<1>();
    }
    __syncthreads();  // every thread's copies are visible to the CTA
    lowrank_slots<NT>(a, sv, b0, nb);
  }
}

// The CTA's partial of z, [8 * NT token rows][64 factor rows], into slot blockIdx.x (the
// first group's contributors are CTAs 0, 1, ...).
template <int NT>
__device__ __forceinline__ void lowrank_piece(const DecodeJob& a) {
  __syncthreads();  // every warp's running sums are in shared memory
  for (int it = threadIdx.x; it < 512 * NT; it += kThreads) {
    const int L = it & 31, j = (it >> 5) & 3, mnt = it >> 7, nt = mnt % NT, m = mnt / NT;
    float z = 0.f;
#pragma unroll
    for (int s = 0; s < 4; ++s) z += lds_f32(a.zacc + (uint32_t)((((m * 4 + s) * NT + nt) * 4 + j) * 32 + L) * 4u);
    const int q = 16 * m + (L >> 2) + 8 * (j >> 1), row = 8 * nt + 2 * (L & 3) + (j & 1);
    if (VQ3_IN(((size_t)blockIdx.x * 8 * NT + row) * 64 + q, (size_t)a.max_pieces * 512 * NT, 21))
      __stcg(a.lr_z + ((size_t)blockIdx.x * 8 * NT + row) * 64 + q, z);
  }
}

// ------------------------------------------------------------------ decode

// A fragment of k-step S, 16-channel tile M, from the lane's string.
template <int F, int S, int M>
__device__ __forceinline__ void a_frag(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase, uint32_t (&a)[4]) {
  if constexpr (Fmt<F>::kVec == 2) {
    // one index per output pair: entry = (channel 2p, channel 2p+1)
    constexpr int n0 = (S * 4 + M) * 4;
    const uint32_t l0 = lut(lut_addr<F, n0 + 0>(w, lanebase));
    const uint32_t l1 = lut(lut_addr<F, n0 + 1>(w, lanebase));
    const uint32_t l2 = lut(lut_addr<F, n0 + 2>(w, lanebase));
    const uint32_t l3 = lut(lut_addr<F, n0 + 3>(w, lanebase));
    a[0] = __byte_perm(l0, l1, 0x5410);  // row g   (channel 2p):   inputs k, k+1
    a[1] = __byte_perm(l0, l1, 0x7632);  // row g+8 (channel 2p+1): inputs k, k+1
    a[2] = __byte_perm(l2, l3, 0x5410);  // row g:   inputs k+8, k+9
    a[3] = __byte_perm(l2, l3, 0x7632);  // row g+8: inputs k+8, k+9
  } else {
    // one index per weight, index (e, c) at n0 + 2e + c: entry = the weight in the low half
    constexpr int n0 = (S * 4 + M) * 8;
    uint32_t l[8];
    l[0] = lut(lut_addr<F, n0 + 0>(w, lanebase));
    l[1] = lut(lut_addr<F, n0 + 1>(w, lanebase));
    l[2] = lut(lut_addr<F, n0 + 2>(w, lanebase));
    l[3] = lut(lut_addr<F, n0 + 3>(w, lanebase));
    l[4] = lut(lut_addr<F, n0 + 4>(w, lanebase));
    l[5] = lut(lut_addr<F, n0 + 5>(w, lanebase));
    l[6] = lut(lut_addr<F, n0 + 6>(w, lanebase));
    l[7] = lut(lut_addr<F, n0 + 7>(w, lanebase));
    a[0] = __byte_perm(l[0], l[2], 0x5410);  // row g   (channel 2p):   inputs k, k+1
    a[1] = __byte_perm(l[1], l[3], 0x5410);  // row g+8 (channel 2p+1): inputs k, k+1
    a[2] = __byte_perm(l[4], l[6], 0x5410);  // row g:   inputs k+8, k+9
    a[3] = __byte_perm(l[5], l[7], 0x5410);  // row g+8: inputs k+8, k+9
  }
}

template <int F, int S, int M, int NT>
__device__ __forceinline__ void mma_step(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase,
                                         float (&acc)[4][NT][4], const uint32_t (&b)[NT][8]) {
  uint32_t a[4];
  a_frag<F, S, M>(w, lanebase, a);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) mma16816(acc[M][nt], a, b[nt][2 * S], b[nt][2 * S + 1]);
}

template <int F, int S, int NT>
__device__ __forceinline__ void kstep(const uint32_t (&w)[Fmt<F>::kWords], uint32_t lanebase,
                                      float (&acc)[4][NT][4], const uint32_t (&b)[NT][8]) {
  mma_step<F, S, 0, NT>(w, lanebase, acc, b);
  mma_step<F, S, 1, NT>(w, lanebase, acc, b);
  mma_step<F, S, 2, NT>(w, lanebase, acc, b);
  mma_step<F, S, 3, NT>(w, lanebase, acc, b);
}

// One super-unit: the lane's index string from its ring slot, the B fragments
// of stage slot p (NT KB at xb, chunks swizzled by p & 7).
template <int F, int NT>
__device__ __forceinline__ void compute_cell(uint32_t slot, uint32_t xb, int lane, int swz, uint32_t lanebase,
                                             float (&acc)[4][NT][4]) {
  uint32_t w[Fmt<F>::kWords];
#pragma unroll
  for (int q = 0; q < FmtSizes<F>::kChunks; ++q) {
    const uint4 v = lds128(slot + (uint32_t)(q * 512 + lane * 16));
    w[4 * q + 0] = v.x;
    w[4 * q + 1] = v.y;
    w[4 * q + 2] = v.z;
    w[4 * q + 3] = v.w;
  }
  uint32_t b[NT][8];
  const uint32_t lo = (uint32_t)((lane ^ swz) * 16);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 v = lds128(xb + (uint32_t)((nt * 2 + h) * 512) + lo);
      b[nt][4 * h + 0] = v.x;
      b[nt][4 * h + 1] = v.y;
      b[nt][4 * h + 2] = v.z;
      b[nt][4 * h + 3] = v.w;
    }
  kstep<F, 0, NT>(w, lanebase, acc, b);
  kstep<F, 1, NT>(w, lanebase, acc, b);
  kstep<F, 2, NT>(w, lanebase, acc, b);
  kstep<F, 3, NT>(w, lanebase, acc, b);
}

// Lane-private tables: entry k of matrix t replicated into words k*32 .. k*32+31
// at tab + t * stride, written 4 lanes (16 bytes) at a time. A vector format's
// codebook word k is (component 0 | component 1 << 16); a scalar entry is
// stored as (entry | entry << 16). The codebook loads go out at kernel start and
// the stores follow the first rotation, so that their latencies overlap.
template <int F>
struct TableLoad {
  static constexpr int E = Fmt<F>::kEntries;
  static constexpr int kItems = 3 * E * 8;
  static constexpr int kPer = (kItems + kThreads - 1) / kThreads;
  const uint32_t* cb[3];
  uint32_t v[kPer];
  __device__ void load(const uint32_t* cb0, const uint32_t* cb1, const uint32_t* cb2) {
    cb[0] = cb0;
    cb[1] = cb1;
    cb[2] = cb2;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = threadIdx.x + r * kThreads;
      const int t = i / (E * 8), k = (i >> 3) % E;
      const uint32_t* p = t == 0 ? cb[0] : (t == 1 ? cb[1] : cb[2]);
      v[r] = 0u;
      if (i < kItems && p) {
        if constexpr (Fmt<F>::kVec == 2) {
          v[r] = __ldg(p + k);
        } else {
          const uint32_t h = __ldg(reinterpret_cast<const uint16_t*>(p) + k);
          v[r] = h | (h << 16);
        }
      }
    }
  }
  __device__ void store(uint32_t tab) const {
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = threadIdx.x + r * kThreads;
      const int t = i / (E * 8), k = (i >> 3) % E, q = i & 7;
      const uint32_t* p = t == 0 ? cb[0] : (t == 1 ? cb[1] : cb[2]);
      if (i < kItems && p) sts128(tab + (uint32_t)(t * Tab<F>::kStride + k * 128 + q * 16), v[r], v[r], v[r], v[r]);
    }
  }
};

// Index-copy cursor of one warp: the next cell of its CTA's range whose copies
// are to be issued. All of it advances by increments; the group-dependent parts
// are recomputed only when a group ends.
struct Cursor {
  const uint4* src;  // this lane's first 16 bytes of the warp's segment SU in the next cell
  int left;          // cells of the range not yet issued
  int kg_left;       // column groups left in the current group (including the next cell)
  int g;             // group of the next cell
  uint32_t slot;     // ring slot of the next copy: byte offset
  bool live;         // the warp's segment exists in group g
#ifdef VQ3_BOUNDS_CHECK
  const uint4* base;  // the matrix's packed indices and their extent in 16-byte units
  size_t extent;
#endif
};

constexpr int kSlots = 3;
// A warp's ring: kSlots slots of one super-unit each.
template <int F>
struct Ring {
  static constexpr int kSlotBytes = FmtSizes<F>::kSuBytes;
  static constexpr int kWarpBytes = kSlots * kSlotBytes;
};

__device__ __forceinline__ void cell_range(const DecodeJob& a, int& c0, int& c1) {
  c0 = a.c0;
  c1 = a.c1;
}

// The job's cell range of this CTA.
__device__ __forceinline__ void set_range(DecodeJob& a) {
  const int cells = a.cells();
  a.c0 = range_begin_w(cells, a.grid, blockIdx.x, a.n_kg(), a.lw);
  a.c1 = range_begin_w(cells, a.grid, blockIdx.x + 1, a.n_kg(), a.lw);
}

// Points the cursor at column group kg of group g.
template <int F>
__device__ __forceinline__ void cursor_group(const DecodeJob& a, Cursor& cur, int g, int kg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sg = g * kWarps + warp;
  const int n_kg = a.n_kg();
  cur.g = g;
  cur.kg_left = n_kg - kg;
  cur.live = sg < a.n_seg();
  const bool two = a.n_mats > 1;
  const int mat = two ? (sg & 1) : 0;
  const int mg = two ? (sg >> 1) : sg;
  cur.src = (mat ? a.packed1 : a.packed0) + ((size_t)mg * n_kg + kg) * FmtSizes<F>::kSuUint4 + lane;
#ifdef VQ3_BOUNDS_CHECK
  cur.base = mat ? a.packed1 : a.packed0;
  cur.extent = (size_t)(a.d_out / kSuChannels) * n_kg * FmtSizes<F>::kSuUint4;
#endif
}

// Issues the index copies of the warp's segment in the cursor's next cell (an
// empty commit group past the range end or for a segment past the last).
template <int F>
__device__ __forceinline__ void issue_cell(const DecodeJob& a, Cursor& cur, uint32_t ring_lane) {
  if (cur.left > 0 && cur.live) {
    const uint32_t s = ring_lane + cur.slot;
#pragma unroll
    for (int q = 0; q < FmtSizes<F>::kChunks; ++q)
#ifdef VQ3_BOUNDS_CHECK
      if (VQ3_IN(cur.src + 32 * q - cur.base, cur.extent, 1))
#endif
        cp_async16(s + (uint32_t)(q * 512), cur.src + 32 * q);
  }
  cp_async_commit();
  constexpr uint32_t kSlot = (uint32_t)Ring<F>::kSlotBytes;
  cur.slot = cur.slot == (kSlots - 1) * kSlot ? 0u : cur.slot + kSlot;
  cur.src += FmtSizes<F>::kSuUint4;
  --cur.left;
  if (--cur.kg_left == 0 && cur.left > 0) cursor_group<F>(a, cur, cur.g + 1, 0);
}

// Index copies of the first n cells of the CTA's range.
template <int F>
__device__ __forceinline__ Cursor decode_begin(const DecodeJob& a, const SmemView& sv, int n) {
  Cursor cur{nullptr, 0, 0, 0, 0u, false};
  if ((int)blockIdx.x >= a.grid) return cur;
  int c0, c1;
  cell_range(a, c0, c1);
  cur.left = (int)(c1 - c0);
  cursor_group<F>(a, cur, c0 / a.n_kg(), c0 % a.n_kg());
  const uint32_t ring_lane = sv.ring + (uint32_t)((threadIdx.x >> 5) * Ring<F>::kWarpBytes + (threadIdx.x & 31) * 16);
  for (int k = 0; k < n; ++k) issue_cell<F>(a, cur, ring_lane);
  return cur;
}

// Decodes the CTA's range of cells; `cur` has issued the copies of its first
// 1 .. kSlots cells, the rest of the prologue follows the first stage.
// LR: a linear layer with low-rank factors (its CTAs of the first segment group also form z).
template <int F, int NT, typename T, bool LR>
__device__ __forceinline__ void decode_run(const DecodeJob& a, const T* src, Cursor& cur, const SmemView& sv,
                                           const TableLoad<F>* tables, int* status) {
  constexpr int PIECE = 512 * NT;
  constexpr int KS = StageCfg<NT>::kSlots;
  if ((int)blockIdx.x >= a.grid) {  // uniform over the CTA
    if (tables) tables->store(sv.tab);  // for a later job; its first barrier orders them
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_kg = a.n_kg(), n_seg = a.n_seg();
  int c0, c1;
  cell_range(a, c0, c1);
  const uint32_t ring = sv.ring + (uint32_t)(warp * Ring<F>::kWarpBytes);
  constexpr uint32_t kSlot = (uint32_t)Ring<F>::kSlotBytes;
  const uint32_t ring_lane = ring + (uint32_t)(lane * 16);
  const bool two = a.n_mats > 1;
  uint32_t use_slot = 0;  // ring slot of the next cell to compute
  int issued = (int)(c1 - c0) - cur.left;  // copies issued so far (the prologue)
  int g = c0 / n_kg, kg = c0 % n_kg;  // group and column group of the next cell
  float acc[4][NT][4];
  uint32_t lane_base = 0;
  bool live = false;
  int sg = 0;
  const int total = (int)(c1 - c0);
  int first = 1;  // the next cell starts the range's part of a group
  if constexpr (LR && NT <= 2) {
    if (c0 < n_kg) {  // this warp's running sums of z start at zero
#pragma unroll
      for (int k = 0; k < NT * 4; ++k) sts_f32(a.zacc + (uint32_t)((warp * NT * 4 + k) * 32 + lane) * 4u, 0.f);
    }
  }
  for (int r0 = 0; r0 < total; r0 += KS) {
    const int kg_s = kg;  // column group of the round's first cell
    const int len = total - r0 < KS ? total - r0 : KS;
    if (a.ready) {
      // the chunks of the round's column groups must be complete
      if (tid == 0) {
        const int ckg = a.chunk / kSuInputs;
        const int lg = __ffs(ckg) - 1;
        const Window win(kg_s, len, lg, n_kg >> lg);
        for (int i = 0; i < win.n; ++i) poll_geq(a.ready + win.chunk(i), a.ready_target, status);
      }
      __syncthreads();  // thread 0's acquire loads, then the barrier: the chunks are visible to the CTA
    }
    stage_round<NT, T>(a, src, kg_s, len, sv);
    if (tables && r0 == 0) tables->store(sv.tab);  // ordered before the decode by the barrier below
    for (; issued < kSlots; ++issued) issue_cell<F>(a, cur, ring_lane);  // rest of the prologue
    // the round's cells of the first segment group (cell index = column group there)
    const int n0 = (LR && NT <= 2 && c0 + r0 < n_kg) ? min(len, n_kg - (c0 + r0)) : 0;
    __syncthreads();
    if constexpr (LR) {
      if (n0) lr_copy(a, sv, c0 + r0, min(n0, kLrBatch));  // lands while the first cell is decoded
    }
    for (int p = 0; p < len; ++p) {
      if (first) {  // the range's part of group g starts
        sg = g * kWarps + warp;
        live = sg < n_seg;
        lane_base = a.tab | (uint32_t)(lane * 4) | ((two && (sg & 1)) ? Tab<F>::kStride : 0u);
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[m][nt][j] = 0.f;
      }
      cp_async_wait<kSlots - 1>();  // this cell's index copies have landed
      if (live)
        compute_cell<F, NT>(ring + use_slot, sv.stage + (uint32_t)(p * NT * 1024), lane, p & 7, lane_base, acc);
      issue_cell<F>(a, cur, ring_lane);  // refill the slot just read, kSlots cells ahead
      if constexpr (LR && NT <= 2) {
        if (n0 && p == 0) {
          // z's share of the round's first-group cells (the stage holds them all; the factor
          // copies issued before the loop have landed while the first cell was decoded): early,
          // so that z is complete well before the segment groups are; where the CTA's part of
          // the first group ends in this round, its partial of z
          lr_round<NT>(a, sv, c0 + r0, n0);
          if ((c1 < n_kg ? c1 : n_kg) <= c0 + r0 + len) {
            lowrank_piece<NT>(a);
            signal(a.lr_done, nullptr);
          }
        }
      }
      use_slot = use_slot == (kSlots - 1) * kSlot ? 0u : use_slot + kSlot;
      first = (++kg == n_kg);
      if (first || r0 + p + 1 == total) {
        // this warp's segment over the range's part of group g: one piece
        if (live) {
          const int piece = blockIdx.x - cta_of_w(g * n_kg, a.cells(), a.grid, n_kg, a.lw);
          float* pc = a.pieces + ((size_t)sg * a.max_pieces + piece) * PIECE;
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (VQ3_IN(pc - a.pieces + ((m * NT + nt) * 4 + j) * 32 + lane, (size_t)n_seg * a.max_pieces * PIECE, 8))
                  __stcg(pc + ((m * NT + nt) * 4 + j) * 32 + lane, acc[m][nt][j]);
        }
        signal(a.group_done + g, nullptr);
      }
      if (first) {
        kg = 0;
        ++g;
      }
    }
    __syncthreads();  // every warp is done with the stage
  }
  cp_async_wait<0>();
  __syncthreads();
}

// ------------------------------------------------------------------ SwiGLU and output tasks

// SwiGLU tasks: one per 64 intermediate channels mg, h = silu(s_g g) * (s_u u)
// for the pass's rows as fp32 into hbuf [rows][d_inter]; a CTA takes mg and
// mg + grid together so that their loads overlap. Each task counts itself done
// in its h chunk's word.
template <int NT>
__device__ __forceinline__ void swiglu_tasks(const PersistArgs& a, const DecodeJob& gu, unsigned* h_done,
                                             int* status) {
  constexpr int PIECE = 512 * NT;
  constexpr int P = 8;
  const int n_mg = a.d_inter / kSuChannels;
  const int per_chunk = a.h_chunk / kSuChannels;
  const int G = gridDim.x;
  for (int m0 = blockIdx.x; m0 < n_mg; m0 += 2 * G) {
    const int m1 = m0 + G;
    const bool two = m1 < n_mg;
    const int g0 = (2 * m0) / kWarps, g1 = two ? (2 * m1) / kWarps : g0;  // groups of segments 2m, 2m+1
    const int n0 = gu.contributors(g0), n1 = two ? gu.contributors(g1) : 0;
    // the scales are inputs: their loads go out before the wait
    float sc[NT][2][2];
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      int r, c;
      item_pos<NT>(q * 512 + threadIdx.x, r, c);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int ch = (k && two ? m1 : m0) * kSuChannels + c;
        const bool sok = VQ3_IN(ch, a.d_inter, 10);
        sc[q][k][0] = sok ? __half2float(__ushort_as_half(__ldg(a.gate.scales + ch))) : 0.f;
        sc[q][k][1] = sok ? __half2float(__ushort_as_half(__ldg(a.up.scales + ch))) : 0.f;
      }
    }
    if (threadIdx.x == 0) {
      if (VQ3_IN(gu.group_done + g0 - a.ctl, a.n_ctl, 26)) poll_geq(gu.group_done + g0, (unsigned)n0, status);
      if (two && VQ3_IN(gu.group_done + g1 - a.ctl, a.n_ctl, 26)) poll_geq(gu.group_done + g1, (unsigned)n1, status);
    }
    __syncthreads();  // thread 0's acquire loads, then the barrier: the pieces are visible to the CTA
    const float* pg0 = gu.seg_pieces(2 * m0, PIECE);
    const float* pu0 = gu.seg_pieces(2 * m0 + 1, PIECE);
    const float* pg1 = gu.seg_pieces(2 * m1 - (two ? 0 : 2 * G), PIECE);  // unused unless two
    const float* pu1 = pg1 + (size_t)gu.max_pieces * PIECE;
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      const int it = q * 512 + threadIdx.x;
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      const int nmax = n0 > n1 ? n0 : n1;
      for (int q0 = 0; q0 < nmax; q0 += P) {
        float v[4][P];
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const size_t o = it + (size_t)(q0 + j) * PIECE;
          const size_t ext = (size_t)gu.n_seg() * gu.max_pieces * PIECE;
          v[0][j] = (q0 + j < n0 && VQ3_IN(pg0 - gu.pieces + o, ext, 9)) ? __ldcg(pg0 + o) : 0.f;
          v[1][j] = (q0 + j < n0 && VQ3_IN(pu0 - gu.pieces + o, ext, 9)) ? __ldcg(pu0 + o) : 0.f;
          v[2][j] = (q0 + j < n1 && VQ3_IN(pg1 - gu.pieces + o, ext, 9)) ? __ldcg(pg1 + o) : 0.f;
          v[3][j] = (q0 + j < n1 && VQ3_IN(pu1 - gu.pieces + o, ext, 9)) ? __ldcg(pu1 + o) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < P; ++j) {
          s[0] += v[0][j];
          s[1] += v[1][j];
          s[2] += v[2][j];
          s[3] += v[3][j];
        }
      }
      int r, c;
      item_pos<NT>(it, r, c);
      if (r < a.rows) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (k == 1 && !two) break;
          const int ch = (k ? m1 : m0) * kSuChannels + c;
          if (VQ3_IN((size_t)r * a.d_inter + ch, (size_t)8 * NT * a.d_inter, 11))
            __stcg(a.hbuf + (size_t)r * a.d_inter + ch, silu_f(sc[q][k][0] * s[2 * k]) * (sc[q][k][1] * s[2 * k + 1]));
        }
      }
    }
    const bool hok = VQ3_IN(h_done + m0 / per_chunk - a.ctl, a.n_ctl, 27) &&
                     (!two || VQ3_IN(h_done + m1 / per_chunk - a.ctl, a.n_ctl, 27));
    if (hok) signal(h_done + m0 / per_chunk, two ? h_done + m1 / per_chunk : nullptr);
    else __syncthreads();  // (a bounds-check build's skip keeps the barrier count of signal)
  }
}

// U z for one output task with factors, on the tensor cores: the task's items form four
// (16-channel tile m, 8-row tile nt) accumulator tiles; warp w takes tile w >> 2 over
// factors 16 (w & 3) .. + 15, with U's rows (channel pairs 2 (8m + g), + 1, as the pieces
// pair them) as A and z as B, split as z = hi + lo in FP16 (two MMAs, ~22 bits of z).
// Each warp writes its partial tile to yp [4 tiles][4 k-steps][4][32] (FP32).
template <int NT>
__device__ __forceinline__ void lowrank_out_mma(int part, int rank, uint32_t ur, const float* zs, float* yp) {
  constexpr int kZs = 68;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int tl = warp >> 2, s = warp & 3;
  const int mnt = part * 4 + tl, m = mnt / NT, nt = mnt % NT;
  const int q0 = 16 * s + 2 * t;  // factor of b0 / a0 (q0 + 8: b1 / a2)
  const uint32_t r0 = ur + (uint32_t)(16 * m + 2 * g) * 144u + (uint32_t)q0 * 2u;  // channel 2 (8m + g)
  uint32_t a[4];
  a[0] = q0 < rank ? lds32(r0) : 0u;
  a[1] = q0 < rank ? lds32(r0 + 144u) : 0u;  // channel 2 (8m + g) + 1
  a[2] = q0 + 8 < rank ? lds32(r0 + 16u) : 0u;
  a[3] = q0 + 8 < rank ? lds32(r0 + 144u + 16u) : 0u;
  const float* zr = zs + (nt * 8 + g) * kZs + q0;  // token row nt * 8 + g is column g
  const float2 z0 = *reinterpret_cast<const float2*>(zr);
  const float2 z1 = *reinterpret_cast<const float2*>(zr + 8);
  const __half2 h0 = __float22half2_rn(z0), h1 = __float22half2_rn(z1);
  const float2 e0 = __half22float2(h0), e1 = __half22float2(h1);
  const __half2 l0 = __floats2half2_rn(z0.x - e0.x, z0.y - e0.y), l1 = __floats2half2_rn(z1.x - e1.x, z1.y - e1.y);
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  mma16816(c, a, *reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
  mma16816(c, a, *reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
#pragma unroll
  for (int j = 0; j < 4; ++j) yp[((tl * 4 + s) * 4 + j) * 32 + lane] = c[j];
}

// One task per (64 output channels, 8-row tile): out = fp16(scale * sum of pieces).
template <int NT>
__device__ __forceinline__ void output_tasks(const PersistArgs& a, const DecodeJob& j, const SmemView& sv, int* status) {
  constexpr int PIECE = 512 * NT;
  constexpr int P = 32;
  const int n_seg = j.d_out / kSuChannels;
  for (int t = blockIdx.x; t < n_seg * NT; t += gridDim.x) {
    const int sg = t / NT, part = t % NT;
    const int g = sg / kWarps;
    const int count = j.contributors(g);
    // the scale is an input: its load goes out before the wait
    const int it = part * 512 + threadIdx.x;
    int r, c;
    item_pos<NT>(it, r, c);
    const int ch = sg * kSuChannels + c;
    const size_t oext = (size_t)(a.row0 + a.rows) * j.d_out;  // x, out, res_next of the call up to this pass
    const float sc = VQ3_IN(ch, j.d_out, 12) ? __half2float(__ushort_as_half(__ldg(j.scales0 + ch))) : 0.f;
    const float rin = (a.res_next && r < a.rows && VQ3_IN((size_t)(a.row0 + r) * j.d_out + ch, oext, 13))
                          ? load1(a.x + (size_t)(a.row0 + r) * j.d_out + ch) : 0.f;
    if (threadIdx.x == 0) {
      if (VQ3_IN(j.group_done + g - a.ctl, a.n_ctl, 26)) poll_geq(j.group_done + g, (unsigned)count, status);
    }
    __syncthreads();  // as for the SwiGLU tasks
    const float* base = j.seg_pieces(sg, PIECE) + it;
    float y = 0.f;
    for (int q0 = 0; q0 < count; q0 += P) {
      float v[P];
#pragma unroll
      for (int q = 0; q < P; ++q)
        v[q] = (q0 + q < count &&
                VQ3_IN(base - j.pieces + (size_t)(q0 + q) * PIECE, (size_t)n_seg * j.max_pieces * PIECE, 14))
                   ? __ldcg(base + (size_t)(q0 + q) * PIECE) : 0.f;
#pragma unroll
      for (int q = 0; q < P; ++q) y += v[q];
    }
    if (r < a.rows) {
      float v = sc * y;
      const __half o16 = __float2half_rn(v);
      if (VQ3_IN((size_t)(a.row0 + r) * j.d_out + ch, oext, 15)) a.out[(size_t)(a.row0 + r) * j.d_out + ch] = __half_as_ushort(o16);
      if (a.res_next) {
        // the next residual, r + out, and its squares for the partial sums below
        const float rn = round16(rin + __half2float(o16));
        if (VQ3_IN((size_t)(a.row0 + r) * j.d_out + ch, oext, 16))
          a.res_next[(size_t)(a.row0 + r) * j.d_out + ch] = __half_as_ushort(__float2half_rn(rn));
        sv.scratch[r * 64 + c] = __fmul_rn(rn, rn);
      }
    }
    if (a.res_next && a.ss_next) {
      // per row and 16-column group of this task: the squares summed in column order (the
      // group of channel c is its 16-channel MMA tile, so a task holds whole groups)
      __syncthreads();
      const int rr = threadIdx.x >> 2, gq = threadIdx.x & 3;
      const int m_lo = part * 4 / NT, m_hi = (part + 1) * 4 / NT;  // MMA tiles (= groups) of this task
      if (rr < 8 * NT && rr < a.rows && gq >= m_lo && gq < m_hi) {
        float ssum = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) ssum += sv.scratch[rr * 64 + 16 * gq + k];
        if (VQ3_IN((size_t)(a.row0 + rr) * (j.d_out / 16) + sg * 4 + gq, (size_t)(a.row0 + a.rows) * (j.d_out / 16), 17))
          a.ss_next[(size_t)(a.row0 + rr) * (j.d_out / 16) + sg * 4 + gq] = ssum;
      }
      __syncthreads();  // the scratch is reused by the next task
    }
  }
}

// The output tasks of a linear layer with low-rank factors: out = fp16(scale * sum of pieces
// + U z), z summed from the first group's partials in CTA order, then U z on the tensor cores
// with its k-step partials added in order, all before the single rounding. A CTA takes its
// tasks t and t + grid together, so that their loads overlap; the tasks are dealt from the
// last CTA down, so that the CTAs of the first group (which also formed z) take one.
template <int NT>
__device__ __forceinline__ void output_tasks_lr(const PersistArgs& a, const DecodeJob& j, const SmemView& sv, int* status) {
  constexpr int PIECE = 512 * NT;
  constexpr int P = 32;           // piece loads in flight
  constexpr int kZs = 68;         // row stride of z in shared memory: 16-byte rows, banks apart
  const int n_seg = j.d_out / kSuChannels;
  const int n_tasks = n_seg * NT;
  const int G = gridDim.x;
  const int count0 = j.contributors(0);
  // scratch (free in this step): z [8 * NT][kZs] at 16 KB; U's rows of the tasks taken together
  // at 24 KB (task k's 64 channels from k * 64 rows on, 144-byte rows: the channels a warp reads
  // fall on distinct banks); the U z partials of task k at 44 KB + k * 8 KB
  float* zs = sv.scratch + 4096;
  constexpr uint32_t kUs = 144;
  const uint32_t us = static_cast<uint32_t>(__cvta_generic_to_shared(sv.scratch)) + 24u * 1024u;
  float* yp = sv.scratch + 11 * 1024;
  bool have_z = false;  // zs holds z (formed once per CTA, before its first tasks' pieces)
  for (int t0 = G - 1 - (int)blockIdx.x; t0 < n_tasks; t0 += 2 * G) {
    const int nk = t0 + G < n_tasks ? 2 : 1;  // tasks taken together (uniform over the CTA)
    {
      // U's rows, copied while the pieces are awaited (16 bytes per thread and copy; the
      // previous tasks' reads of them ended before the barrier that followed them)
      const int per_row = a.lr_rank / 8;  // 16-byte chunks of a row
      for (int i = threadIdx.x; i < nk * kSuChannels * per_row; i += kThreads) {
        const int row = i / per_row, k = i - row * per_row;  // row: task row >> 6, channel row & 63
        const uint16_t* src = a.lr_u + ((size_t)((t0 + (row >> 6) * G) / NT) * kSuChannels + (row & 63)) * a.lr_rank;
        if (VQ3_IN(src + k * 8 - a.lr_u, (size_t)j.d_out * a.lr_rank, 18))
          cp_async16(us + (uint32_t)row * kUs + (uint32_t)k * 16u, src + k * 8);
      }
      cp_async_commit();
    }
    int sg[2], part[2], cnt[2], r[2], c[2], ch[2];
    float sc[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = (k < nk) ? t0 + k * G : t0;  // a missing second task repeats the first (not stored)
      sg[k] = t / NT;
      part[k] = t % NT;
      cnt[k] = j.contributors(sg[k] / kWarps);
      item_pos<NT>(part[k] * 512 + threadIdx.x, r[k], c[k]);
      ch[k] = sg[k] * kSuChannels + c[k];
      // the scale is an input: its load goes out before the wait
      sc[k] = VQ3_IN(ch[k], j.d_out, 12) ? __half2float(__ushort_as_half(__ldg(j.scales0 + ch[k]))) : 0.f;
    }
    const bool do_z = !have_z;  // the CTA's first tasks also form z
    if (threadIdx.x == 0) {
      if (VQ3_IN(j.group_done + sg[0] / kWarps - a.ctl, a.n_ctl, 26))
        poll_geq(j.group_done + sg[0] / kWarps, (unsigned)cnt[0], status);
      if (nk == 2 && VQ3_IN(j.group_done + sg[1] / kWarps - a.ctl, a.n_ctl, 26))
        poll_geq(j.group_done + sg[1] / kWarps, (unsigned)cnt[1], status);
      if (do_z) poll_geq(j.lr_done, (unsigned)count0, status);  // z's partials
    }
    __syncthreads();  // as for the SwiGLU tasks
    // z[row][q] = the sum of the partials of CTAs 0, 1, ..., count0 - 1 in that order: the
    // loads of its first ZP partials go out together with the pieces' loads below
    constexpr int ZP = NT == 1 ? 16 : 8;
    float zb[NT][ZP];
    if (do_z) {
#pragma unroll
      for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int k = 0; k < ZP; ++k)
          zb[i][k] = (k < count0 && VQ3_IN(threadIdx.x + i * kThreads + (size_t)k * PIECE, (size_t)j.max_pieces * PIECE, 19))
                         ? __ldcg(j.lr_z + threadIdx.x + i * kThreads + (size_t)k * PIECE) : 0.f;
    }
    // both tasks' sums of pieces, each in piece (= CTA) order: the first task's pieces then the
    // second's, loaded P at a time
    float y[2] = {0.f, 0.f};
    {
      const float* b0 = j.seg_pieces(sg[0], PIECE) + part[0] * 512 + threadIdx.x;
      const float* b1 = j.seg_pieces(sg[1], PIECE) + part[1] * 512 + threadIdx.x - (size_t)cnt[0] * PIECE;
      const int tot = cnt[0] + (nk == 2 ? cnt[1] : 0);
      for (int q0 = 0; q0 < tot; q0 += P) {
        float v[P];
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const int i = q0 + q;
          const size_t pext = (size_t)n_seg * j.max_pieces * PIECE;
          v[q] = i < cnt[0] ? (VQ3_IN(b0 - j.pieces + (size_t)i * PIECE, pext, 14) ? __ldcg(b0 + (size_t)i * PIECE) : 0.f)
                            : ((i < tot && VQ3_IN(b1 - j.pieces + (size_t)i * PIECE, pext, 14)) ? __ldcg(b1 + (size_t)i * PIECE) : 0.f);
        }
#pragma unroll
        for (int q = 0; q < P; ++q) {
          if (q0 + q < cnt[0])
            y[0] += v[q];
          else
            y[1] += v[q];
        }
      }
    }
    if (do_z) {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const int e = threadIdx.x + i * kThreads;  // [row][q] of the pass, 64 factors per row
        float z = 0.f;
#pragma unroll
        for (int k = 0; k < ZP; ++k) z += zb[i][k];
        for (int k0 = ZP; k0 < count0; k0 += ZP) {  // more than ZP contributors
          float v[ZP];
#pragma unroll
          for (int k = 0; k < ZP; ++k)
            v[k] = (k0 + k < count0 && VQ3_IN(e + (size_t)(k0 + k) * PIECE, (size_t)j.max_pieces * PIECE, 19))
                       ? __ldcg(j.lr_z + e + (size_t)(k0 + k) * PIECE) : 0.f;
#pragma unroll
          for (int k = 0; k < ZP; ++k) z += v[k];
        }
        zs[(e >> 6) * kZs + (e & 63)] = z;
      }
      have_z = true;
    }
    {
      cp_async_wait<0>();
      __syncthreads();  // z and every thread's copies of U's rows are visible
      lowrank_out_mma<NT>(part[0], a.lr_rank, us, zs, yp);
      if (nk == 2) lowrank_out_mma<NT>(part[1], a.lr_rank, us + 64u * kUs, zs, yp + 2048);
      __syncthreads();  // the U z partials are in shared memory
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (k >= nk) break;
      if (r[k] < a.rows) {
        float v = sc[k] * y[k];
        {
          // low-rank correction: the item's four k-step partials in order (its tile is
          // warp >> 2 of the task, its accumulator register warp & 3)
          const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
          const float* q = yp + k * 2048 + ((warp >> 2) * 16 + (warp & 3)) * 32 + lane;
          v += ((q[0] + q[128]) + q[256]) + q[384];
        }
        const __half o16 = __float2half_rn(v);
        if (VQ3_IN((size_t)(a.row0 + r[k]) * j.d_out + ch[k], (size_t)(a.row0 + a.rows) * j.d_out, 15))
          a.out[(size_t)(a.row0 + r[k]) * j.d_out + ch[k]] = __half_as_ushort(o16);
      }
    }
  }
}

// ------------------------------------------------------------------ the kernel

template <int NT, int F, bool LR = false>
struct Smem {
  static constexpr uint32_t kRing = kWarps * Ring<F>::kWarpBytes;
  static constexpr uint32_t kStage = StageCfg<NT>::kBytes;
  static constexpr uint32_t kScratch = kWarps * 4096;  // rotation scratch, 4 KB per warp
  // running sums of the low-rank projection (linear layers with factors, up to 16 rows):
  // [warp][NT][4][32]
  static constexpr uint32_t kZacc = (LR && NT <= 2) ? (uint32_t)(kWarps * NT * 128 * 4) : 0u;
  static constexpr uint32_t kTabs = 3 * Tab<F>::kStride;  // gate, up, down (or one matrix)
  static constexpr uint32_t kTotal = kRing + kStage + kScratch + kZacc + Tab<F>::kAlign + kTabs;
};

// LR: the instantiation for a linear layer with low-rank factors (up to 16 rows); the others
// carry none of its code.
template <int NT, int F, bool LR>
__global__ void __launch_bounds__(kThreads, 1) persistent_kernel(PersistArgs a) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ int s_flag;
  __shared__ float s_inv[32];  // 1/rms of the pass's rows (pre-norm residual step)
  __shared__ float s_part[32];  // sums of squares of the rows' column ranges
  __shared__ int s_range3[2];   // the down step's cell range
  SmemView sv;
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(dsm));
  sv.ring = base;
  using SM = Smem<NT, F, LR>;
  sv.stage = base + SM::kRing;
  sv.scratch = reinterpret_cast<float*>(dsm + SM::kRing + SM::kStage);
  sv.tab = (base + SM::kRing + SM::kStage + SM::kScratch + SM::kZacc + Tab<F>::kAlign - 1) & ~(Tab<F>::kAlign - 1);
  sv.flag = &s_flag;
  int* status = a.status;
  unsigned* ctl = a.ctl;

  DecodeJob j1;
  j1.d_in = a.d_model;
  j1.d_out = a.mlp ? a.d_inter : a.d_model_out;
  j1.n_mats = a.mlp ? 2 : 1;
  j1.packed0 = a.gate.packed;
  j1.packed1 = a.up.packed;
  j1.scales0 = a.gate.scales;
  j1.pieces = a.pieces1;
  j1.grid = a.grid1;
  j1.max_pieces = a.max_pieces1;
  j1.tab = sv.tab;
  j1.src_ld = (size_t)a.d_model;
  j1.rows = a.rows;
  j1.block = a.block_in;
  j1.scale = a.scale_in;
  j1.chunk = a.x_chunk;
  j1.signs = a.signs_in;
  j1.inv = (!LR && a.norm) ? s_inv : nullptr;
  j1.res_delta = (!LR && a.norm && a.res_delta) ? a.res_delta + (size_t)a.row0 * a.d_model : nullptr;
  j1.ready = nullptr;
  j1.ready_target = 0;
  j1.group_done = ctl + (a.mlp ? a.off_g : a.off_o);
  j1.lr_v = LR ? a.lr_v : nullptr;
  j1.lr_rank = a.lr_rank;
  j1.lr_z = a.lr_z;
  j1.lr_done = ctl + a.off_z;
  j1.lw = LR ? a.lr_lw : 0;
  j1.zacc = base + SM::kRing + SM::kStage + SM::kScratch;
  set_range(j1);
  if (LR && (int)threadIdx.x < NT) {
    // U's rows of this CTA's output tasks (64 channels each), towards L2 (copied from there later)
    const int n_seg = a.d_model_out / kSuChannels;
    for (int t = blockIdx.x; t < n_seg * NT; t += gridDim.x)
      if (t % NT == (int)threadIdx.x)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.lr_u + (size_t)(t / NT) * kSuChannels * a.lr_rank),
                     "r"((uint32_t)(kSuChannels * a.lr_rank * 2)) : "memory");
  }
  if (!LR && a.mlp && threadIdx.x == 0) {  // (the low-rank instantiation serves linear layers only)
    // the down step's cell range, worked out now, away from the hand-off before that step
    const int n_seg3 = a.d_model / kSuChannels;
    const int cells3 = (n_seg3 + kWarps - 1) / kWarps * (a.d_inter / kSuInputs);
    s_range3[0] = range_begin(cells3, a.grid3, blockIdx.x);
    s_range3[1] = range_begin(cells3, a.grid3, blockIdx.x + 1);
  }

  TableLoad<F> tables;
  tables.load(a.gate.codebook, a.mlp ? a.up.codebook : nullptr, a.mlp ? a.down.codebook : nullptr);
  // one cell's index copies, then the rotation of x (its loads not queued behind
  // the bulk of the prologue), then the rest of the prologue
  Cursor cur = decode_begin<F>(j1, sv, 1);
  if (!LR && a.norm && a.ss_in) {
    // the rows' sums of squares from the previous layer's partials (16 columns each): one
    // warp per row, lanes over the partials in a fixed order, then the warp's xor tree
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, n_part = a.d_model / 16;
    for (int rr = warp; rr < a.rows; rr += kWarps) {
      const float* p = a.ss_in + (size_t)(a.row0 + rr) * n_part;
      float ss = 0.f;
      for (int q = lane; q < n_part; q += 32)
        if (VQ3_IN((size_t)(a.row0 + rr) * n_part + q, (size_t)(a.row0 + a.rows) * n_part, 22)) ss += __ldcg(p + q);
#pragma unroll
      for (int h = 16; h > 0; h >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, h);
      if (lane == 0) s_inv[rr] = 1.0f / sqrtf(ss / (float)a.d_model + a.eps);
    }
    __syncthreads();
  } else if (!LR && a.norm) {
    // pre-norm residual step for the pass's rows: r' = fp16(x + delta) over the whole row
    // (every CTA, for its own 1/rms), the 64-column slices s with s % grid == CTA written to
    // res_out. Each row is split into `parts` column ranges, one warp each (parts = warps per
    // row, a power of two); a lane's loads go out four 8-column groups at a time. The sum of
    // squares is reduced in a fixed order: lanes in sequence, the warp's xor tree, parts in order.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, d = a.d_model;
    int parts = 1;
    while (parts * 2 * a.rows <= kWarps) parts *= 2;
    const int n8 = d / 8;
    for (int w = warp; w < a.rows * parts; w += kWarps) {
      const int rr = w / parts, part = w % parts;
      const size_t ro = (size_t)(a.row0 + rr) * d;
      const int g0 = part * n8 / parts, g1 = (part + 1) * n8 / parts;
      float ss = 0.f;
      for (int gb = g0; gb < g1; gb += 4 * 32) {
        uint4 xv[4], dv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int g = gb + u * 32 + lane;
          if (g < g1 && VQ3_IN(ro / 8 + g, (size_t)(a.row0 + a.rows) * d / 8, 23)) {
            xv[u] = __ldg(reinterpret_cast<const uint4*>(a.x + ro) + g);
            if (a.res_delta) dv[u] = __ldg(reinterpret_cast<const uint4*>(a.res_delta + ro) + g);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int g = gb + u * 32 + lane;
          if (g >= g1) break;
          uint4 rv = xv[u];
          if (a.res_delta) {
            const __half2* xh = reinterpret_cast<const __half2*>(&xv[u]);
            const __half2* dh = reinterpret_cast<const __half2*>(&dv[u]);
            __half2* rh = reinterpret_cast<__half2*>(&rv);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 xf = __half22float2(xh[k]), df = __half22float2(dh[k]);
              rh[k] = __floats2half2_rn(xf.x + df.x, xf.y + df.y);
            }
          }
          const __half2* rh = reinterpret_cast<const __half2*>(&rv);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(rh[k]);
            ss = fmaf(f.x, f.x, ss);
            ss = fmaf(f.y, f.y, ss);
          }
          if (a.res_out && (g >> 3) % (int)gridDim.x == (int)blockIdx.x &&
              VQ3_IN(ro / 8 + g, (size_t)(a.row0 + a.rows) * d / 8, 25))
            *(reinterpret_cast<uint4*>(a.res_out + ro) + g) = rv;
        }
      }
#pragma unroll
      for (int h = 16; h > 0; h >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, h);
      if (lane == 0) s_part[w] = ss;
    }
    __syncthreads();
    if ((int)threadIdx.x < a.rows) {
      float ss = 0.f;
      for (int q = 0; q < parts; ++q) ss += s_part[threadIdx.x * parts + q];
      s_inv[threadIdx.x] = 1.0f / sqrtf(ss / (float)d + a.eps);
    }
    __syncthreads();
  }
  decode_run<F, NT, uint16_t, LR>(j1, a.x + (size_t)a.row0 * a.d_model, cur, sv, &tables, status);

  if (!LR && a.mlp) {
    DecodeJob j3;
    j3.d_in = a.d_inter;
    j3.d_out = a.d_model;
    j3.n_mats = 1;
    j3.packed0 = j3.packed1 = a.down.packed;
    j3.scales0 = a.down.scales;
    j3.pieces = a.pieces3;
    j3.grid = a.grid3;
    j3.max_pieces = a.max_pieces3;
    j3.tab = sv.tab + 2u * Tab<F>::kStride;
    j3.src_ld = (size_t)a.d_inter;
    j3.rows = a.rows;
    j3.block = a.block_dn;
    j3.scale = a.scale_dn;
    j3.chunk = a.h_chunk;
    j3.signs = a.signs_dn;
    j3.ready = ctl + a.off_hd;
    j3.ready_target = (unsigned)(a.h_chunk / kSuChannels);
    j3.group_done = ctl + a.off_o;
    j3.lr_v = nullptr;
    j3.lr_rank = 0;
    j3.lr_z = nullptr;
    j3.lr_done = nullptr;
    j3.lw = 0;
    j3.zacc = 0u;
    j3.c0 = s_range3[0];  // written by thread 0 before the first barrier of the gate/up step
    j3.c1 = s_range3[1];
    swiglu_tasks<NT>(a, j1, ctl + a.off_hd, status);
    // one cell's index copies ahead of the h rotation, the rest after it (as for x)
    Cursor cur3 = decode_begin<F>(j3, sv, 1);
    decode_run<F, NT, float, false>(j3, a.hbuf, cur3, sv, nullptr, status);
    output_tasks<NT>(a, j3, sv, status);
  } else if constexpr (LR && NT <= 2) {
    output_tasks_lr<NT>(a, j1, sv, status);
  } else {
    output_tasks<NT>(a, j1, sv, status);
  }

  cp_async_wait<0>();
  // the last CTA to finish clears the counters for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned old;  // acquire and release: every CTA's waits precede the last CTA's clearing
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(ctl) : "memory");
    s_flag = old + 1 == gridDim.x;
  }
  __syncthreads();
  if (s_flag)
    for (int i = threadIdx.x; i < a.n_ctl; i += kThreads) ctl[i] = 0u;
}

// Every format's kernel needs more than half an SM's shared memory: one CTA per SM,
// so the grid (and the workspace sized from it) is the same for all formats.
static_assert(2 * Smem<1, VQ3_FORMAT_2X16>::kTotal > 228 * 1024, "one CTA per SM");
static_assert(Smem<4, VQ3_FORMAT_LUT4>::kTotal <= 227 * 1024 && Smem<4, VQ3_FORMAT_2X64>::kTotal <= 227 * 1024 &&
                  Smem<2, VQ3_FORMAT_LUT4, true>::kTotal <= 227 * 1024 &&
                  Smem<2, VQ3_FORMAT_2X64, true>::kTotal <= 227 * 1024,
              "shared memory per CTA");

template <int NT, int F, bool LR>
cudaError_t launch_nt(const PersistArgs& a, cudaStream_t st) {
  const int smem = (int)Smem<NT, F, LR>::kTotal;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(persistent_kernel<NT, F, LR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, persistent_kernel<NT, F, LR>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int NT>
int occupancy() {
  using K = Smem<NT, VQ3_FORMAT_2X64>;
  int n = 0;
  if (cudaFuncSetAttribute(persistent_kernel<NT, VQ3_FORMAT_2X64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)K::kTotal) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, persistent_kernel<NT, VQ3_FORMAT_2X64, false>, kThreads, K::kTotal) !=
          cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n > 0 ? n : 1;
}

}  // namespace

int dec_tiles_per_pass(int rows) { return rows <= 8 ? 1 : (rows <= 16 ? 2 : 4); }

int persist_grid(int nt) {
  static int cache[64][3] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return device_sm_count();
  }
  const int slot = nt == 1 ? 0 : (nt == 2 ? 1 : 2);
  if (!cache[dev][slot]) {
    const int occ = nt == 1 ? occupancy<1>() : (nt == 2 ? occupancy<2>() : occupancy<4>());
    const int g = occ * device_sm_count();
    cache[dev][slot] = g > kDecMaxGrid ? kDecMaxGrid : g;
  }
  return cache[dev][slot];
}

int persist_decode_grid(int d_in, int d_out, int n_mats, int grid) {
  const int n_seg = (d_out / kSuChannels) * n_mats;
  const long long cells = (long long)((n_seg + kDecWarps - 1) / kDecWarps) * (d_in / kSuInputs);
  return cells < grid ? (int)cells : grid;  // every decoding CTA owns at least one cell
}

bool persist_cells_fit(int d_in, int d_out, int n_mats, int grid) {
  const long long n_seg = (long long)(d_out / kSuChannels) * n_mats;
  const long long cells = (n_seg + kDecWarps - 1) / kDecWarps * (d_in / kSuInputs);
  return cells * grid < (1ll << 32);  // the kernel's cell arithmetic is 32-bit unsigned
}

int persist_max_pieces(int d_in, int d_out, int n_mats, int grid, int lw) {
  const long long n_kg = d_in / kSuInputs;
  const long long n_seg = (long long)(d_out / kSuChannels) * n_mats;
  const long long n_grp = (n_seg + kDecWarps - 1) / kDecWarps;
  const long long cells = n_grp * n_kg;
  // the kernel's partition (cta_of_w), in 64-bit here
  auto cost = [&](long long x) { return 8 * x + lw * (x < n_kg ? x : n_kg); };
  auto cta = [&](long long x) { return lw ? ((cost(x) + 1) * grid - 1) / cost(cells) : ((x + 1) * grid - 1) / cells; };
  int best = 1;
  for (long long s = 0; s < n_grp; ++s) {
    const long long b0 = cta(s * n_kg), b1 = cta(s * n_kg + n_kg - 1);
    if (b1 - b0 + 1 > best) best = (int)(b1 - b0 + 1);
  }
  return best;
}

int persist_lowrank_weight(int d_in, int d_out, int grid) {
  // first-group cells weighted 1 + 2/8 when there are at least 4 cells per CTA (so that every
  // CTA keeps a cell) and the kernel's 32-bit partition arithmetic holds
  const long long n_kg = d_in / kSuInputs;
  const long long cells = ((d_out / kSuChannels) + kDecWarps - 1) / kDecWarps * n_kg;
  constexpr int lw = 2;
  if (cells < 4ll * grid) return 0;
  if ((8 * cells + lw * n_kg + 1) * grid >= (1ll << 32)) return 0;
  return lw;
}

int persist_chunk(int d, int block) {
  const int span = block < kSuChannels ? kSuChannels : block;
  int chunk = span;
  while (chunk * 2 <= 1024 && d % (chunk * 2) == 0) chunk *= 2;
  return chunk;
}

namespace {
template <int F>
cudaError_t launch_fmt(const PersistArgs& a, int nt, cudaStream_t st) {
  switch (nt) {
    // a linear layer with low-rank factors has its own instantiation (up to 16 rows)
    case 1: return a.lr_v ? launch_nt<1, F, true>(a, st) : launch_nt<1, F, false>(a, st);
    case 2: return a.lr_v ? launch_nt<2, F, true>(a, st) : launch_nt<2, F, false>(a, st);
    case 4: return a.lr_v ? cudaErrorInvalidValue : launch_nt<4, F, false>(a, st);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_persistent(const PersistArgs& a, int nt, cudaStream_t st) {
  switch (a.format) {
    case VQ3_FORMAT_2X64: return launch_fmt<VQ3_FORMAT_2X64>(a, nt, st);
    case VQ3_FORMAT_2X16: return launch_fmt<VQ3_FORMAT_2X16>(a, nt, st);
    case VQ3_FORMAT_LUT4: return launch_fmt<VQ3_FORMAT_LUT4>(a, nt, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vq3
