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

// Position of index (p, i) in the GPU layout: byte offset of its 16-byte word
// group is not unique (an index may straddle two words), so this returns the
// lane string coordinates instead.
struct LanePos {
  size_t su;  // super-unit number
  int lane;   // 0..31
  int n;      // index number inside the lane string, 0..63
};

inline LanePos lane_pos(int d_in, int p, int i) {
  const int mg = p / 32, pl = p % 32, m = pl / 8, g = pl % 8;
  const int kg = i / 64, il = i % 64, s = il / 16, r = il % 16;
  int t, e;
  if (r < 8) { t = r / 2; e = r % 2; } else { t = (r - 8) / 2; e = 2 + r % 2; }
  LanePos lp;
  lp.su = (size_t)mg * (size_t)(d_in / 64) + (size_t)kg;
  lp.lane = g * 4 + t;
  lp.n = (s * 4 + m) * 4 + e;
  return lp;
}

// Byte offset inside the matrix of 32-bit word w (0..11) of lane L of SU su.
inline size_t lane_word_offset(size_t su, int lane, int w) {
  return su * kSuBytes + (size_t)((w / 4) * 32 + lane) * 16 + (size_t)(w % 4) * 4;
}

// ---------------------------------------------------------------------------
// kernels (launch wrappers; all return cudaGetLastError() after launch)
// ---------------------------------------------------------------------------

struct GemvMat {
  const uint4* packed;
  const uint32_t* codebook;  // [64] FP16x2 words (component 0 in the low half)
  const uint16_t* scales;    // [d_out]
};

enum GemvMode { kModeLinear = 0, kModeSwiglu = 1 };

struct GemvArgs {
  const uint16_t* xr;  // rotated input, FP16 [rows][d_in] (row stride d_in)
  int rows;            // valid rows of this pass (<= 8 * n_tiles)
  int d_in, d_out;
  int kc_len;          // inputs per K chunk (multiple of 64, divides d_in)
  int n_mats;          // 1 (linear) or 2 (gate and up)
  GemvMat mats[2];
  float* partial;      // [n_kc][n_mats][kMaxPassRows][d_out]
  unsigned* counters;  // [d_out / 64], zero on entry, zero on exit
  int mode;
  uint16_t* out;       // FP16 [rows][d_out] (row stride d_out)
};

constexpr int kMaxPassRows = 32;

inline int pick_kc_len(int d_in) {
  for (int c = 1024; c >= 64; c >>= 1)
    if (d_in % c == 0) return c;
  return 0;
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st);
cudaError_t launch_fwht(const uint16_t* x, int rows, int n, int block, const uint32_t* signs,
                        uint16_t* out, cudaStream_t st);
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
