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
// A super-unit (SU) covers 64 output channels (32 output pairs) x 64 input
// columns: 2048 six-bit indices, 1536 bytes. SU (mg, kg) of a matrix starts at
// byte (mg * (d_in/64) + kg) * 1536, so one output group's K range is
// contiguous. Inside an SU, warp lane L (g = L/4, t = L%4) owns 64 indices
// (384 bits = 12 words); its words 4q..4q+3 are the 16 bytes at SU offset
// (q*32 + L)*16, q = 0..2, so each of the three 128-bit loads of a warp reads
// 512 contiguous bytes. Lane index n (bits [6n, 6n+6) of the lane's 384-bit
// string, least significant bit first) is
//     n = (s*4 + m)*4 + e          s: k-step of 16 inputs, m: 16-channel tile
//     pair  p = mg*32 + m*8 + g
//     input i = kg*64 + s*16 + {2t, 2t+1, 2t+8, 2t+9}[e]
// which is exactly what lane L needs for the A fragment of an m16n8k16 MMA
// whose row g is channel 2p and row g+8 is channel 2p+1.
// ---------------------------------------------------------------------------
constexpr int kSuChannels = 64;
constexpr int kSuInputs = 64;
constexpr int kSuBytes = 1536;
constexpr int kSuUint4 = kSuBytes / 16;  // 96

inline bool layout_supported(int d_in, int d_out) {
  return d_in > 0 && d_out > 0 && d_in % kSuInputs == 0 && d_out % kSuChannels == 0;
}

// Byte offset of 32-bit word w (0..11) of lane L's string in SU su.
__host__ __device__ inline size_t lane_word_offset(size_t su, int lane, int w) {
  return su * kSuBytes + (size_t)((w / 4) * 32 + lane) * 16 + (size_t)(w % 4) * 4;
}

// ---------------------------------------------------------------------------
// Rotated activations in "fragment order" (what the decode kernel reads):
// for each 64-input column group kg and each 8-row tile nt, 256 32-bit words
// (1 KB). Lane L = 4g + t needs the FP16 pairs w_v = (x'[8nt+g][kg*64 + 16s +
// 2t + 8hh], x'[8nt+g][... + 1]), v = 2s + hh (s = 0..3, hh = 0..1): the B
// fragments of four m16n8k16 MMAs. They are stored as two 16-byte chunks per
// lane, chunk h = v/4 of lane L at tile offset (h*32 + L)*16, so a warp's two
// 128-bit loads each read 512 contiguous bytes without bank conflicts. Rows
// past the last valid row are zero.
// ---------------------------------------------------------------------------
__host__ __device__ inline size_t frag_half_index(int row, int col, int n_tiles) {
  const int kg = col / 64, cl = col % 64, s = cl / 16, r = cl % 16;
  const int hh = r / 8, t = (r % 8) / 2, half = r % 2;
  const int nt = row / 8, g = row % 8;
  const int lane = 4 * g + t, v = 2 * s + hh;
  const size_t word = ((size_t)kg * n_tiles + nt) * 256 + (size_t)((v / 4) * 32 + lane) * 4 + (v % 4);
  return word * 2 + half;
}

inline int row_tiles(int rows) { return (rows + 7) / 8; }

// ---------------------------------------------------------------------------
// kernels (launch wrappers; all return cudaGetLastError() after launch)
// ---------------------------------------------------------------------------

enum MatMode { kModeLinear = 0, kModeSwiglu = 1 };

struct DecMat {
  const uint4* packed;
  const uint32_t* codebook;  // [64] FP16x2 words (component 0 in the low half)
  const uint16_t* scales;    // [d_out]
};

// One launch of the decode kernel over row tiles [nt0, nt0 + NT) of the input:
// writes the per-segment partial sums ("pieces"); a combine kernel finishes.
struct DecArgs {
  const uint32_t* xfrag;  // rotated input in fragment order, n_tiles row tiles
  int n_tiles;            // row tiles of xfrag (all rows)
  int nt0;                // first row tile of this pass
  int d_in, d_out;        // per matrix
  int n_mats;             // 1 (linear) or 2 (gate and up, interleaved segments)
  DecMat mats[2];
  float* pieces;          // [n_segments][max_pieces][512 * NT] partial sums
  int grid, max_pieces;
  int ksplit;             // warps per segment inside a CTA
  int* status;            // device status word (set to 2 if the lookup tables are misplaced)
};

// Where the pieces of a decode launch are and how many CTAs contributed.
struct PieceMap {
  const float* pieces;
  int n_kg;               // 64-input column groups of d_in
  int n_mats;
  int n_groups;           // segment groups
  int seg_per_group;      // kDecWarps / ksplit
  int grid, max_pieces;
  int nt;                 // row tiles per piece (NT)
};

// Sums gate and up pieces, h = silu(s_g*g) * (s_u*u), rotates h by the down
// projection's Hadamard blocks (signs) and writes h' in fragment order.
struct SwigluRotateArgs {
  PieceMap pm;
  const uint16_t* scale_gate;
  const uint16_t* scale_up;
  int d_inter;            // intermediate width (gate/up d_out)
  int rows;               // valid rows of the pass
  int row0;               // first row of the pass
  int block;              // down rotation block
  const uint32_t* signs;  // down signs or null
  uint32_t* hfrag;        // output, fragment order, n_tiles row tiles
  int n_tiles;
};

// Sums pieces, y = scale * sum, writes FP16 rows [row0, row0 + rows) of out.
struct LinearOutArgs {
  PieceMap pm;
  const uint16_t* scales;
  int d_out;
  int rows, row0;
  uint16_t* out;          // row-major [*][d_out]
};

cudaError_t launch_swiglu_rotate(const SwigluRotateArgs& a, cudaStream_t st);
cudaError_t launch_linear_out(const LinearOutArgs& a, cudaStream_t st);

constexpr int kDecWarps = 16;  // warps per decode CTA = segments per group
constexpr int kDecMaxGrid = 2048;

int device_sm_count();
int dec_tiles_per_pass(int rows);  // 1, 2 or 4 row tiles (8, 16 or 32 rows)
int dec_ksplit(int d_in, int d_out, int n_mats);  // warps per segment inside a CTA (power of two)
int dec_groups(int d_in, int d_out, int n_mats);  // segment groups (kDecWarps / ksplit segments each)
int dec_grid(int d_in, int d_out, int n_mats);  // never more CTAs than cells
int dec_max_pieces(int d_in, int d_out, int n_mats, int grid);
cudaError_t launch_decode(const DecArgs& a, int nt, cudaStream_t st);
// One pass (up to 32 rows) of the MLP block, or of a single linear layer, as
// one persistent cooperative kernel. Its steps (decode gate/up, SwiGLU, decode
// down, output) hand over through counters in `ctl` rather than grid barriers;
// the rotations happen inside the decode steps.
struct PersistArgs {
  const uint16_t* x;        // row-major [*][d_model]
  int row0, rows;           // rows of this pass: [row0, row0 + rows), rows <= 8 * NT
  int mlp;                  // 1: MLP block (gate, up, down); 0: one linear layer (gate)
  int d_model, d_inter;     // MLP: hidden and intermediate widths; linear: d_model = d_in
  int d_model_out;          // linear: d_out
  int block_in, block_dn;   // rotation blocks of the gate/up (or linear) input and of the down input
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
  int* status;              // workspace status word (3: a wait timed out)
  uint16_t* out;            // row-major [*][d_model] (linear: [*][d_out])
};

int persist_grid(int nt);  // CTAs of the persistent kernel: resident CTAs per SM x SMs
int persist_decode_grid(int d_in, int d_out, int n_mats, int grid);  // decoding CTAs (<= cells)
int persist_max_pieces(int d_in, int d_out, int n_mats, int grid);
int persist_chunk(int d, int block);  // rotation chunk: whole blocks, up to 1024 columns
cudaError_t launch_persistent(const PersistArgs& a, int nt, cudaStream_t st);

cudaError_t launch_fwht(const uint16_t* x, int rows, int n, int block, const uint32_t* signs,
                        uint16_t* out, cudaStream_t st);
// Same rotation, written in fragment order (rows padded with zeros to 8 * n_tiles).
cudaError_t launch_fwht_frag(const uint16_t* x, int rows, int n, int block, const uint32_t* signs,
                             uint32_t* xfrag, int n_tiles, cudaStream_t st);
cudaError_t launch_residual_rmsnorm(uint16_t* resid, const uint16_t* delta, int rows, int n,
                                    float eps, uint16_t* normed, cudaStream_t st);
cudaError_t launch_dequant(const vq3_linear& L, int apply_scale, uint16_t* w_out, cudaStream_t st);

// Byte range of the arrival counters inside an MLP workspace laid out for `rows`.
void mlp_counter_range(int rows, const vq3_mlp_layer* layer, size_t* offset, size_t* bytes);

// Checks the arguments of an MLP call except the workspace (status as the entry points).
int mlp_validate(const uint16_t* x, int rows, const vq3_mlp_layer* layer, const uint16_t* out);

// Records the thread-local error message and returns `code`.
int set_error(int code, const char* fmt, ...);

}  // namespace vq3
