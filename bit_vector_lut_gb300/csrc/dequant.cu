// Debug/test kernel: dense weights from the GPU index layout, any index format.
// w_out[o][i] = C[idx][c] (apply_scale = 0) or fp16(fp32(scale[o]) * fp32(C[idx][c])), where
// idx is the index of output group o / v (v = 2 for the vector formats: channel
// o is component c = o % 2 of pair o / 2; v = 1 for the scalar format: c = 0).
// Source of the weight definition: model card "anemll/anemll-forge-qwen3.8-27B",
// section "Release 0.2: three-bit MLP, token-mixer rotations, distilled weights",
// bullet "Three bits per MLP weight", and the release-comparison table (two-bit
// vector LUT 2x16, four-bit LUT).
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
namespace {

__global__ void dequant_kernel(const uint8_t* __restrict__ packed, const uint16_t* __restrict__ codebook,
                               const uint16_t* __restrict__ scales, int d_in, int d_out, int apply_scale,
                               int format, uint16_t* __restrict__ w_out) {
  const int nb = format == VQ3_FORMAT_2X64 ? 6 : 4;
  const int vec = format == VQ3_FORMAT_LUT4 ? 1 : 2;
  const int su_bytes = (format == VQ3_FORMAT_2X64 ? 3 : (format == VQ3_FORMAT_2X16 ? 2 : 4)) * 512;
  const long long total = (long long)d_out * d_in;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int o = (int)(e / d_in), i = (int)(e % d_in);
    // inverse of the super-unit mapping (see vq3_internal.h)
    const int mg = o / 64, ol = o % 64, pl = ol / 2, c = ol % 2;
    const int m = pl / 8, g = pl % 8;
    const int kg = i / 64, il = i % 64, s = il / 16, r = il % 16;
    const int t = (r < 8) ? (r >> 1) : ((r - 8) >> 1);
    const int ee = (r < 8) ? (r & 1) : (2 + (r & 1));
    const int lane = g * 4 + t;
    const int n0 = (s * 4 + m) * 4 + ee;
    const int n = vec == 1 ? 2 * n0 + c : n0;
    const size_t su = (size_t)mg * (d_in / 64) + kg;
    const int bit = nb * n, wd = bit / 32, off = bit % 32;
    const uint8_t* base = packed + su * su_bytes;
    uint64_t v = *reinterpret_cast<const uint32_t*>(base + (size_t)((wd / 4) * 32 + lane) * 16 + (wd % 4) * 4);
    if (off + nb > 32) {
      const int w1 = wd + 1;
      v |= (uint64_t)(*reinterpret_cast<const uint32_t*>(base + (size_t)((w1 / 4) * 32 + lane) * 16 + (w1 % 4) * 4))
           << 32;
    }
    const int k = (int)((v >> off) & ((1u << nb) - 1u));
    const uint16_t cv = vec == 1 ? codebook[k] : codebook[2 * k + c];
    uint16_t out = cv;
    if (apply_scale) {
      const float f = __half2float(__ushort_as_half(scales[o])) * __half2float(__ushort_as_half(cv));
      out = __half_as_ushort(__float2half_rn(f));
    }
    w_out[(size_t)o * d_in + i] = out;
  }
}

}  // namespace

cudaError_t launch_dequant(const vq3_linear& L, int apply_scale, uint16_t* w_out, cudaStream_t st) {
  const long long total = (long long)L.d_out * L.d_in;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  dequant_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint8_t*>(L.packed), L.codebook, L.scales,
                                                  L.d_in, L.d_out, apply_scale, L.format, w_out);
  return cudaGetLastError();
}

}  // namespace vq3
