// vq3_mlp_forward_noalloc: the MLP block with its scratch in a fixed device array.
//
// Some callers cannot call cudaMalloc: a plugin running inside a host framework
// that owns every device allocation, a serving process that reserved its whole
// memory budget up front, or code that must not allocate while another thread
// captures a CUDA graph. For them this entry point takes the scratch that
// vq3_mlp_forward reads from a caller workspace out of the file-scope array
// below instead. The array is part of the library's device image: every GPU
// that loads this module holds it until the process exits.
#include <mutex>

#include "vq3_internal.h"

namespace vq3 {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)VQ3_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace vq3

using namespace vq3;

extern "C" int vq3_mlp_forward_noalloc(const uint16_t* x, int rows, const vq3_mlp_layer* layer, uint16_t* out,
                                       void* stream) {
  int rc = mlp_validate(x, rows, layer, out);
  if (rc) return rc;
  if (rows == 0) return set_error(VQ3_OK, "");
  // the largest pass (32, 16 or 8 rows) whose scratch fits the array; more rows run as more passes
  int cap = 0;
  size_t need = 0;
  for (int c = 32; c >= 8; c /= 2) {
    need = mlp_workspace_bytes_capped(rows, layer, c);
    if (need <= kNoAllocScratchBytes) {
      cap = c;
      break;
    }
  }
  if (!cap)
    return set_error(VQ3_ENOSPACE,
                     "mlp_noalloc: a %d/%d block needs %zu bytes of scratch even in 8-row passes, more than "
                     "the fixed %zu-byte array (VQ3_NOALLOC_SCRATCH_BYTES); use vq3_mlp_forward with a workspace",
                     layer->gate.d_in, layer->gate.d_out, need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return set_error(VQ3_ECUDA, "mlp_noalloc: cudaGetSymbolAddress: %s (%s)", cudaGetErrorName(e),
                     cudaGetErrorString(e));
  // The array keeps the previous call's contents. The status word (offset 0) and the
  // counter words after it must start at zero: one clear covers both, so a wait that
  // gave up in an earlier call does not make this call skip its waits.
  size_t off = 0, bytes = 0;
  mlp_counter_range(layer, &off, &bytes);
  e = cudaMemsetAsync(scratch, 0, off + bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return set_error(VQ3_ECUDA, "mlp_noalloc: clearing the status and counter words: %s (%s)", cudaGetErrorName(e),
                     cudaGetErrorString(e));
  return mlp_forward_capped(x, rows, layer, out, scratch, kNoAllocScratchBytes, stream, cap);
}

extern "C" int vq3_noalloc_status(int* status_host, void* stream) {
  if (!status_host) return set_error(VQ3_EINVAL, "noalloc_status: null pointer");
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(status_host, scratch, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess)
    return set_error(VQ3_ECUDA, "noalloc_status: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
  return set_error(VQ3_OK, "");
}
