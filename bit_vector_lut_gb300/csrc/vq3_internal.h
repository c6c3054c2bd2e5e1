// Internal declarations of the VQ3 library: GPU index layout, launch helpers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/vq3.h"

namespace vq3 {

// ---------------------------------------------------------------------------
// GPU index layout ("super-units").
//
// A super-unit (SU) covers 64 output channels x 64 input columns. SU (mg, kg)
// of a matrix starts at byte (mg * (d_in/64) + kg) * SU bytes, so one output
// group's K range is contiguous. Inside an SU, warp lane L (g = L/4, t = L%4)
// owns a string of W 32-bit words (its indices, least significant bit first);
// words 4q..4q+3 are the 16 bytes at SU offset (q*32 + L)*16, so each 128-bit
// load of a warp reads 512 contiguous bytes. With index width b, index n of
// the string sits at bits [b n, b n + b). For the vector formats (one index per
// output pair) the lane holds 64 indices,
//     n = (s*4 + m)*4 + e          s: k-step of 16 inputs, m: 16-channel tile
//     pair  p = mg*32 + m*8 + g
//     input i = kg*64 + s*16 + {2t, 2t+1, 2t+8, 2t+9}[e]
// and for the scalar format (one index per weight) 128 indices,
//     n = ((s*4 + m)*4 + e)*2 + c, channel 2p + c, p and i as above,
// which is what lane L needs for the A fragment of an m16n8k16 MMA whose row g
// is channel 2p and row g+8 is channel 2p+1.
//   format  b  indices/lane  W   SU bytes
//   2x64    6  64            12  1536
//   2x16    4  64             8  1024
//   lut4    4  128           16  2048
// ---------------------------------------------------------------------------
constexpr int kSuChannels = 64;
constexpr int kSuInputs = 64;
constexpr int kSuBytes = 1536;           // the three-bit format's SU
constexpr int kSuUint4 = kSuBytes / 16;  // 96
constexpr int kMaxSuBytes = 2048;

template <int F>
struct Fmt;
template <>
struct Fmt<VQ3_FORMAT_2X64> {
  static constexpr int kBits = 6, kVec = 2, kEntries = 64, kWords = 12;
};
template <>
struct Fmt<VQ3_FORMAT_2X16> {
  static constexpr int kBits = 4, kVec = 2, kEntries = 16, kWords = 8;
};
template <>
struct Fmt<VQ3_FORMAT_LUT4> {
  static constexpr int kBits = 4, kVec = 1, kEntries = 16, kWords = 16;
};
// Derived sizes: 16-byte chunks per lane string, SU bytes and uint4s, indices per lane string.
template <int F>
struct FmtSizes {
  static constexpr int kChunks = Fmt<F>::kWords / 4;
  static constexpr int kSuBytes = kChunks * 512;
  static constexpr int kSuUint4 = kSuBytes / 16;
  static constexpr int kIndices = 128 / Fmt<F>::kVec;
};

inline bool format_supported(int f) { return f == VQ3_FORMAT_2X64 || f == VQ3_FORMAT_2X16 || f == VQ3_FORMAT_LUT4; }
inline int format_bits(int f) { return f == VQ3_FORMAT_2X64 ? 6 : 4; }
inline int format_vec(int f) { return f == VQ3_FORMAT_LUT4 ? 1 : 2; }
inline int format_words(int f) { return f == VQ3_FORMAT_2X64 ? 12 : (f == VQ3_FORMAT_2X16 ? 8 : 16); }
inline int format_su_bytes(int f) { return format_words(f) / 4 * 512; }

inline bool layout_supported(int d_in, int d_out) {
  return d_in > 0 && d_out > 0 && d_in % kSuInputs == 0 && d_out % kSuChannels == 0;
}

// Byte offset of 32-bit word w of lane L's string in SU su (three-bit format).
__host__ __device__ inline size_t lane_word_offset(size_t su, int lane, int w) {
  return su * kSuBytes + (size_t)((w / 4) * 32 + lane) * 16 + (size_t)(w % 4) * 4;
}
// The same for an SU of su_bytes bytes.
__host__ __device__ inline size_t lane_word_offset(size_t su, int lane, int w, int su_bytes) {
  return su * su_bytes + (size_t)((w / 4) * 32 + lane) * 16 + (size_t)(w % 4) * 4;
}

// ---------------------------------------------------------------------------
// kernels (launch wrappers; all return cudaGetLastError() after launch)
// ---------------------------------------------------------------------------

struct DecMat {
  const uint4* packed;
  const uint32_t* codebook;  // [entries] FP16x2 words (component 0 in the low half); [16] FP16 for lut4
  const uint16_t* scales;    // [d_out]
};

constexpr int kDecWarps = 16;  // warps per decoding CTA = segments per group
constexpr int kDecMaxGrid = 2048;

int device_sm_count();

// ---------------------------------------------------------------------------
// Bounds-check build (-DVQ3_BOUNDS_CHECK): an instrumented global access checks its element
// index against the extent of the buffer it addresses, VQ3_IN(index, extent, site); a
// violation skips the access and is counted in a per-file device record with the first
// site (file id << 8 | site). Each instrumented file defines its record with
// VQ3_BOUNDS_RECORD(name) inside namespace vq3; vq3_bounds_check collects them. In other
// builds VQ3_IN is `true` and nothing is recorded.
#ifdef VQ3_BOUNDS_CHECK
__device__ inline bool vq3_in_bounds(size_t i, size_t n, unsigned site, unsigned* rec) {
  if (i < n) return true;
  if (atomicAdd(&rec[0], 1u) == 0u) atomicExch(&rec[1], site);
  return false;
}
#define VQ3_BOUNDS_RECORD(name)                                                            \
  namespace {                                                                              \
  __device__ unsigned g_bounds[2];                                                         \
  }                                                                                        \
  cudaError_t bounds_read_##name(unsigned* host, bool reset) {                             \
    cudaError_t e = cudaMemcpyFromSymbol(host, g_bounds, sizeof(g_bounds));                \
    if (e == cudaSuccess && reset) {                                                       \
      const unsigned z[2] = {0u, 0u};                                                      \
      e = cudaMemcpyToSymbol(g_bounds, z, sizeof(z));                                      \
    }                                                                                      \
    return e;                                                                              \
  }
#define VQ3_IN(idx, n, site) vq3_in_bounds((size_t)(idx), (size_t)(n), (unsigned)(site), g_bounds)
cudaError_t bounds_read_persistent(unsigned* host, bool reset);
cudaError_t bounds_read_lowrank(unsigned* host, bool reset);
cudaError_t bounds_read_delta(unsigned* host, bool reset);
cudaError_t bounds_read_rotate(unsigned* host, bool reset);
cudaError_t bounds_read_prefill(unsigned* host, bool reset);
cudaError_t bounds_read_prefill_wide(unsigned* host, bool reset);
#else
#define VQ3_BOUNDS_RECORD(name)
#define VQ3_IN(idx, n, site) ((void)(n), true)  // the extent is used only by the check
#endif
// The C ABI's thread-local error message, for host code outside api.cu: report_error sets it
// (printf format) and returns code; report_ok clears it and returns VQ3_OK.
int report_error(int code, const char* fmt, ...);
int report_ok();
int dec_tiles_per_pass(int rows);  // 8-row tiles per pass: 1, 2 or 4 (8, 16 or 32 rows)
// One pass (up to 32 rows) of the MLP block, or of a single linear layer, as
// one persistent cooperative kernel. Its steps (decode gate/up, SwiGLU, decode
// down, output) hand over through counters in `ctl` rather than grid barriers;
// the rotations happen inside the decode steps.
struct PersistArgs {
  const uint16_t* x;        // row-major [*][d_model]
  int row0, rows;           // rows of this pass: [row0, row0 + rows), rows <= 8 * NT
  int mlp;                  // 1: MLP block (gate, up, down); 0: one linear layer (gate)
  int format;               // VQ3_FORMAT_* of every matrix
  // low-rank correction U (V x') of a linear layer (null lr_v: none; MLP: none). The CTAs
  // that decode the first segment group also form z = V x' from their rotated activations
  // and write one partial [8 * NT][64] FP32 each to lr_z; the output step sums them in CTA
  // order and adds U z before rounding.
  const uint16_t* lr_v;     // [lr_rank][d_model], FP16
  const uint16_t* lr_u;     // [d_model_out][lr_rank], FP16
  int lr_rank;              // a multiple of 8, <= 64
  float* lr_z;              // max_pieces1 x [8 * NT][64] FP32
  int lr_lw;                // the first group's cell weight in the CTA ranges (persist_lowrank_weight)
  // pre-norm residual step fused ahead of the block (MLP only): the block's input rows are
  // fp16(r' / sqrt(mean(r'^2) + eps)) with r' = fp16(x + res_delta) (x alone when res_delta is
  // null), and r' is written to res_out (which aliases neither x nor res_delta)
  int norm;
  const uint16_t* res_delta;
  uint16_t* res_out;        // may be null: r' is then not written
  float eps;
  // the residual stack chained by sums of squares (MLP only, norm set, res_delta null):
  // ss_in (or null) holds the rows' sums of squares as FP32 partials per 16 columns,
  // [rows][d / 16], in place of reading the rows; the output step also writes
  // res_next = fp16(x + out) and its partials ss_next in the same layout
  const float* ss_in;
  uint16_t* res_next;
  float* ss_next;
  int d_model, d_inter;     // MLP: hidden and intermediate widths; linear: d_model = d_in
  int d_model_out;          // linear: d_out
  int block_in, block_dn;   // rotation blocks of the gate/up (or linear) input and of the down input
  float scale_in, scale_dn; // 1 / sqrt(block), rounded as the float expression 1.0f / sqrtf(block)
  const uint32_t* signs_in; // sign bits or null
  const uint32_t* signs_dn;
  int x_chunk, h_chunk;     // columns per rotation chunk of x and of h (whole blocks, <= 1024)
  DecMat gate, up, down;
  float* hbuf;              // h of this pass before rotation, fp32 [8 * NT][d_inter] (MLP only)
  float* pieces1;           // split-K partial sums of the gate/up (or linear) decode
  float* pieces3;           // same for down
  int grid;                 // CTAs (all co-resident)
  int grid1, max_pieces1;   // decode grid and piece slots per segment: gate/up (or linear)
  int grid3, max_pieces3;   // same for down
  unsigned* ctl;            // n_ctl counter words, zero before and after every launch
  int n_ctl;
  int off_g, off_hd, off_o; // word offsets: gate/up segment groups, h chunks (SwiGLU tasks
                            // done), output segment groups; word 0 counts finished CTAs
  int off_z;                // linear layer: CTAs whose partial of z (low-rank) is written
  int* status;              // workspace status word (3: a wait timed out)
  uint16_t* out;            // row-major [*][d_model] (linear: [*][d_out])
};

int persist_grid(int nt);  // CTAs of the persistent kernel: resident CTAs per SM x SMs
int persist_decode_grid(int d_in, int d_out, int n_mats, int grid);  // decoding CTAs (<= cells)
int persist_max_pieces(int d_in, int d_out, int n_mats, int grid, int lw = 0);
// Extra weight (eighths of a cell) of the first segment group's cells in the decode kernel's CTA
// ranges for a linear layer with low-rank factors (those CTAs also form z), or 0.
int persist_lowrank_weight(int d_in, int d_out, int grid);
// Whether the decode kernel's 32-bit cell arithmetic holds (cells x grid < 2^32).
bool persist_cells_fit(int d_in, int d_out, int n_mats, int grid);
int persist_chunk(int d, int block);  // rotation chunk: whole blocks, up to 1024 columns
cudaError_t launch_persistent(const PersistArgs& a, int nt, cudaStream_t st);

// Column order of the tensor-core GEMM's activation operand. The GEMM keeps its decoded
// weight tiles in tensor memory, written by tcgen05.st 16x256b: there the K pairs of each
// 16-input group sit in the column order (0, 4, 1, 5, 2, 6, 3, 7), so the activations (the
// other operand) carry the same order: input pair c of a 16-column group is stored at pair
// position 2c (c < 4) or 2(c - 4) + 1. The contraction over K is unchanged.
__host__ __device__ inline int mma_order_col(int col) {
  const int c = (col & 15) >> 1;
  const int pos = c < 4 ? 2 * c : 2 * (c - 4) + 1;
  return (col & ~15) | (pos << 1) | (col & 1);
}
// Input column held at stored column `col` of a row in that order (the inverse map).
__host__ __device__ inline int mma_order_input(int col) {
  const int pos = (col & 15) >> 1;
  const int c = (pos >> 1) + 4 * (pos & 1);
  return (col & ~15) | (c << 1) | (col & 1);
}

// mma_order: store the rotated rows in the GEMM's operand order (mma_order_col); n % 16 == 0.
cudaError_t launch_fwht(const uint16_t* x, int rows, int n, int block, const uint32_t* signs,
                        uint16_t* out, cudaStream_t st, int mma_order = 0);
// Same rotation of FP32 rows, written as FP16.
cudaError_t launch_fwht_f32(const float* x, int rows, int n, int block, const uint32_t* signs, uint16_t* out,
                            cudaStream_t st, int mma_order = 0);

// One VQ3 matrix (or the gate/up pair) against rotated FP16 activations on
// tcgen05 tensor cores: out16 = fp16(s0 * W0 x') for one matrix, or, with
// swiglu, out32 = silu(s0 * W0 x') * (s1 * W1 x') in FP32 (W0 gate, W1 up).
struct PrefillArgs {
  const uint16_t* x;       // rotated activations, FP16 [rows][d_in], 16-byte aligned
  int rows, d_in, d_out;   // d_out: output channels (swiglu: the intermediate width)
  int swiglu;
  int format;              // VQ3_FORMAT_* of W0 (and W1)
  const uint4* packed0;    // GPU-layout indices of W0 (and W1)
  const uint4* packed1;
  const uint32_t* cb0;     // codebooks
  const uint32_t* cb1;
  const uint16_t* scale0;  // per-output-channel scales
  const uint16_t* scale1;
  uint16_t* out16;         // [rows][d_out] FP16 (no swiglu)
  float* out32;            // [rows][d_out] FP32 (swiglu)
  int* status;             // status word (3: a wait timed out)
  const float* lr_y;       // low-rank correction U V x' [rows][d_out] FP32 (no swiglu), or null
  float* part;             // split-tile sums, one 128 x tile-rows FP32 slot per CTA
  unsigned* flags;         // one word per CTA, zero between calls: its slot is filled
  long long work;          // (tile, K step) pairs; set by launch_prefill_gemm
};
// Two tensor-core GEMM kernels serve the many-row path. Up to kPrefillNarrowRows rows:
// launch_prefill_gemm, output tiles of 64 or 128 rows, 4 or 2 tiles per K step sharing one
// activation tile, the decoded weights in tensor memory, activations in the operand order of
// mma_order_col. Above: launch_prefill_wide_gemm, tiles of 256 rows, the decoded weights in
// shared memory, activations in their natural order.
constexpr int kPrefillNarrowRows = 128;
inline bool prefill_wide(int rows) { return rows > kPrefillNarrowRows; }
long long prefill_wide_work(int rows, int d_in, int d_out, int swiglu);
int prefill_wide_grid(int rows, int d_in, int d_out, int swiglu);
cudaError_t launch_prefill_wide_gemm(const PrefillArgs& a, cudaStream_t st);
int prefill_tile_rows(int rows);  // rows per output tile of launch_prefill_gemm: 64 or 128
long long prefill_work(int rows, int d_in, int d_out, int swiglu);
int prefill_max_grid();           // most CTAs of one launch (one per SM)
int prefill_grid(int rows, int d_in, int d_out, int swiglu);
size_t prefill_part_bytes(int rows);  // size of PrefillArgs::part (serves both kernels)
cudaError_t launch_prefill_gemm(const PrefillArgs& a, cudaStream_t st);
// r_next = fp16(r + d), ss[row][g] = sum of r_next^2 over columns 16g .. 16g+15 (or none: ss null).
cudaError_t launch_residual_add_ss(const uint16_t* r, const uint16_t* d, uint16_t* r_next, float* ss, int rows,
                                   int n, cudaStream_t st);
cudaError_t launch_residual_rmsnorm(uint16_t* resid, const uint16_t* delta, int rows, int n,
                                    float eps, uint16_t* normed, cudaStream_t st);
// The same with the updated residual written to resid_out (may equal resid_in).
cudaError_t launch_residual_rmsnorm2(const uint16_t* resid_in, const uint16_t* delta, uint16_t* resid_out, int rows,
                                     int n, float eps, uint16_t* normed, cudaStream_t st);
cudaError_t launch_dequant(const vq3_linear& L, int apply_scale, uint16_t* w_out, cudaStream_t st);
// Gated delta-rule token mixer over blocks of 8 tokens (layouts as vq3_delta_rule_forward).
cudaError_t launch_delta_rule(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* beta,
                              const float* alpha, int tokens, int heads, int d_k, int d_v, float* state,
                              uint16_t* out, cudaStream_t st);
// ylr[r][o] = sum_j U[o][j] z[r][j], z[r][j] = sum_i V[j][i] xr[r][i] (FP32) for the low-rank
// correction (V [rank][d_in], U [d_out][rank] FP16); the projection's sums over
// lowrank_chunks(d_in, rows) input splits go through part [splits][rows][rank], then z
// [rows][rank] after them: lowrank_part_floats(d_in, rows, rank) floats in all.
int lowrank_chunks(int d_in, int rows);
size_t lowrank_part_floats(int d_in, int rows, int rank);
// xr_mma_order: the rows of xr are stored in the GEMM's operand order (mma_order_col).
cudaError_t launch_lowrank(const uint16_t* xr, int rows, int d_in, const uint16_t* V, const uint16_t* U, int rank,
                           int d_out, float* part, float* ylr, cudaStream_t st, int xr_mma_order = 0);

// vq3_mlp_forward with passes of at most `pass_cap` rows (8, 16 or 32), and its
// workspace size; vq3_mlp_forward itself uses 32.
size_t mlp_workspace_bytes_capped(int rows, const vq3_mlp_layer* layer, int pass_cap);
int mlp_forward_capped(const uint16_t* x, int rows, const vq3_mlp_layer* layer, uint16_t* out, void* workspace,
                       size_t ws_bytes, void* stream, int pass_cap);

// Byte range of the counter words inside an MLP workspace (the same for every row count).
void mlp_counter_range(const vq3_mlp_layer* layer, size_t* offset, size_t* bytes);

// Checks the arguments of an MLP call except the workspace (status as the entry points).
int mlp_validate(const uint16_t* x, int rows, const vq3_mlp_layer* layer, const uint16_t* out);

// Records the thread-local error message and returns `code`.
int set_error(int code, const char* fmt, ...);

}  // namespace vq3
