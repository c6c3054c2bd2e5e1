// Debug/test kernel: dense weights from the GPU index layout.
// w_out[2p+c][i] = C[idx[p][i]][c] (apply_scale = 0) or fp16(fp32(scale[2p+c]) * fp32(C[...][c])).
// Source of the weight definition: model card "anemll/anemll-forge-qwen3.8-27B",
// section "Release 0.2: three-bit MLP, token-mixer rotations, distilled weights",
// bullet "Three bits per MLP weight".
#include <cuda_fp16.h>

#include "vq3_internal.h"

namespace vq3 {
namespace {

__global__ void dequant_kernel(const uint8_t* __restrict__ packed, const uint16_t* __restrict__ codebook,
                               const uint16_t* __restrict__ scales, int d_in, int d_out, int apply_scale,
                               uint16_t* __restrict__ w_out) {
  const long long total = (long long)(d_out / 2) * d_in;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(e / d_in), i = (int)(e % d_in);
    // inverse of the super-unit mapping (see vq3_internal.h)
    const int mg = p / 32, pl = p % 32, m = pl / 8, g = pl % 8;
    const int kg = i / 64, il = i % 64, s = il / 16, r = il % 16;
    const int t = (r < 8) ? (r >> 1) : ((r - 8) >> 1);
    const int ee = (r < 8) ? (r & 1) : (2 + (r & 1));
    const int lane = g * 4 + t;
    const int n = (s * 4 + m) * 4 + ee;
    const size_t su = (size_t)mg * (d_in / 64) + kg;
    const int bit = 6 * n, wd = bit / 32, off = bit % 32;
    const uint32_t* w0 = reinterpret_cast<const uint32_t*>(packed + su * kSuBytes + (size_t)((wd / 4) * 32 + lane) * 16) + (wd % 4);
    uint64_t v = *w0;
    if (off + 6 > 32) {
      const int w1i = wd + 1;
      const uint32_t* w1 = reinterpret_cast<const uint32_t*>(packed + su * kSuBytes + (size_t)((w1i / 4) * 32 + lane) * 16) + (w1i % 4);
      v |= (uint64_t)(*w1) << 32;
    }
    const int k = (int)((v >> off) & 63u);
    for (int c = 0; c < 2; ++c) {
      const uint16_t cv = codebook[2 * k + c];
      uint16_t o = cv;
      if (apply_scale) {
        const float f = __half2float(__ushort_as_half(scales[2 * p + c])) * __half2float(__ushort_as_half(cv));
        o = __half_as_ushort(__float2half_rn(f));
      }
      w_out[(size_t)(2 * p + c) * d_in + i] = o;
    }
  }
}

}  // namespace

cudaError_t launch_dequant(const vq3_linear& L, int apply_scale, uint16_t* w_out, cudaStream_t st) {
  const long long total = (long long)(L.d_out / 2) * L.d_in;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  dequant_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint8_t*>(L.packed), L.codebook, L.scales,
                                                  L.d_in, L.d_out, apply_scale, w_out);
  return cudaGetLastError();
}

}  // namespace vq3
