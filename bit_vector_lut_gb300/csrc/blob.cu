// Packed-weight blob of one VQ3 matrix: host-side save and load (the layout is described
// with vq3_blob_write in include/vq3.h). Host code only; it allocates no device memory.
#include <cstring>
#include <vector>

#include "vq3_internal.h"

namespace vq3 {
namespace {

constexpr char kMagic[8] = {'V', 'Q', '3', 'B', 'L', 'O', 'B', '1'};
constexpr uint32_t kVersion = 1;
constexpr size_t kHeaderBytes = 256;
constexpr size_t kAlign = 256;
enum Section { kCanon, kPacked, kScales, kCodebook, kSigns, kU, kV, kSections };

// Little-endian on both the build and the GPU machines' hosts (x86-64, AArch64).
struct Header {
  char magic[8];
  uint32_t version;
  uint32_t header_bytes;
  int32_t d_in, d_out, block, format, lr_rank;
  uint32_t flags;  // bit 0: sign bits present
  uint64_t offset[8];
  uint64_t size[8];
  uint64_t hash;   // FNV-1a 64 of bytes [header_bytes, total)
  uint64_t total;
  uint8_t pad[kHeaderBytes - 40 - 128 - 16];
};
static_assert(sizeof(Header) == kHeaderBytes, "blob header size");

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool pow2_in(int b, int lo, int hi) { return b >= lo && b <= hi && (b & (b - 1)) == 0; }

size_t codebook_bytes(int format) {
  switch (format) {
    case VQ3_FORMAT_2X64: return 64 * 4;
    case VQ3_FORMAT_2X16: return 16 * 4;
    case VQ3_FORMAT_LUT4: return 16 * 2;
    default: return 0;
  }
}

// FNV-1a, 64-bit (offset basis 14695981039346656037, prime 1099511628211).
uint64_t fnv1a64(const uint8_t* p, size_t n) {
  uint64_t h = 14695981039346656037ull;
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;
  }
  return h;
}

// Section sizes and offsets for a descriptor; false if it is unsupported (the message is set).
bool plan(int d_in, int d_out, int format, int lr_rank, int has_signs, Header& h) {
  if (!format_supported(format)) {
    report_error(VQ3_EUNSUPPORTED, "blob: unknown index format %d", format);
    return false;
  }
  if (!layout_supported(d_in, d_out)) {
    report_error(VQ3_EUNSUPPORTED, "blob: d_in=%d and d_out=%d must be positive multiples of 64", d_in, d_out);
    return false;
  }
  if (lr_rank < 0 || lr_rank > 64 || lr_rank % 8) {
    report_error(VQ3_EUNSUPPORTED, "blob: lr_rank=%d must be 0 or a multiple of 8 up to 64", lr_rank);
    return false;
  }
  const size_t idx = vq3_packed_bytes_fmt(format, d_in, d_out);
  h.size[kCanon] = idx;
  h.size[kPacked] = idx;
  h.size[kScales] = (size_t)d_out * 2;
  h.size[kCodebook] = codebook_bytes(format);
  h.size[kSigns] = has_signs ? (size_t)d_in / 32 * 4 : 0;
  h.size[kU] = (size_t)d_out * lr_rank * 2;
  h.size[kV] = (size_t)lr_rank * d_in * 2;
  h.size[7] = 0;
  size_t off = kHeaderBytes;
  for (int s = 0; s < 8; ++s) {
    h.offset[s] = off;
    off = align_up(off + h.size[s]);
  }
  h.total = off;
  return true;
}

}  // namespace
}  // namespace vq3

using namespace vq3;

extern "C" {

size_t vq3_blob_bytes(int d_in, int d_out, int format, int lr_rank, int has_signs) {
  Header h{};
  if (!plan(d_in, d_out, format, lr_rank, has_signs ? 1 : 0, h)) return 0;
  return h.total;
}

int vq3_blob_write(int d_in, int d_out, int block, int format, const uint8_t* canonical, const uint16_t* scales,
                   const void* codebook, const uint32_t* signs, int lr_rank, const uint16_t* lr_u,
                   const uint16_t* lr_v, void* out, size_t out_bytes) {
  if (!canonical || !scales || !codebook || !out) return report_error(VQ3_EINVAL, "blob_write: null pointer");
  if (lr_rank > 0 && (!lr_u || !lr_v)) return report_error(VQ3_EINVAL, "blob_write: null low-rank factors");
  Header h{};
  if (!plan(d_in, d_out, format, lr_rank, signs ? 1 : 0, h)) return VQ3_EUNSUPPORTED;  // message set by plan
  if (!pow2_in(block, 2, 1024) || d_in % block)
    return report_error(VQ3_EUNSUPPORTED, "blob_write: block=%d must be a power of two in [2, 1024] dividing d_in=%d",
                        block, d_in);
  if (out_bytes < h.total) return report_error(VQ3_ENOSPACE, "blob_write: %zu bytes < %zu", out_bytes, (size_t)h.total);
  memcpy(h.magic, kMagic, 8);
  h.version = kVersion;
  h.header_bytes = (uint32_t)kHeaderBytes;
  h.d_in = d_in;
  h.d_out = d_out;
  h.block = block;
  h.format = format;
  h.lr_rank = lr_rank;
  h.flags = signs ? 1u : 0u;
  uint8_t* b = static_cast<uint8_t*>(out);
  memset(b, 0, h.total);  // the alignment gaps are zero, so the hash is a function of the contents
  memcpy(b + h.offset[kCanon], canonical, h.size[kCanon]);
  const int rc = vq3_pack_layout_fmt(format, canonical, d_in, d_out, b + h.offset[kPacked]);
  if (rc) return rc;
  memcpy(b + h.offset[kScales], scales, h.size[kScales]);
  memcpy(b + h.offset[kCodebook], codebook, h.size[kCodebook]);
  if (signs) memcpy(b + h.offset[kSigns], signs, h.size[kSigns]);
  if (lr_rank > 0) {
    memcpy(b + h.offset[kU], lr_u, h.size[kU]);
    memcpy(b + h.offset[kV], lr_v, h.size[kV]);
  }
  h.hash = fnv1a64(b + kHeaderBytes, h.total - kHeaderBytes);
  memcpy(b, &h, kHeaderBytes);
  return report_ok();
}

int vq3_blob_read(const void* blob, size_t bytes, vq3_blob_view* view) {
  if (!blob || !view) return report_error(VQ3_EINVAL, "blob_read: null pointer");
  if (bytes < kHeaderBytes) return report_error(VQ3_EINVAL, "blob_read: %zu bytes, shorter than the header", bytes);
  const uint8_t* b = static_cast<const uint8_t*>(blob);
  Header h;
  memcpy(&h, b, kHeaderBytes);
  if (memcmp(h.magic, kMagic, 8) != 0) return report_error(VQ3_EINVAL, "blob_read: not a VQ3 blob (magic)");
  if (h.version != kVersion || h.header_bytes != kHeaderBytes)
    return report_error(VQ3_EINVAL, "blob_read: version %u, header %u bytes (this library reads version %u)", h.version,
                        h.header_bytes, kVersion);
  Header want{};
  if (!plan(h.d_in, h.d_out, h.format, h.lr_rank, (int)(h.flags & 1u), want))
    return report_error(VQ3_EINVAL, "blob_read: unsupported descriptor (%s)", vq3_last_error());
  if (h.flags & ~1u) return report_error(VQ3_EINVAL, "blob_read: unknown flags 0x%x", h.flags);
  if (!pow2_in(h.block, 2, 1024) || h.d_in % h.block)
    return report_error(VQ3_EINVAL, "blob_read: block=%d does not fit d_in=%d", h.block, h.d_in);
  for (int s = 0; s < 8; ++s)
    if (h.offset[s] != want.offset[s] || h.size[s] != want.size[s])
      return report_error(VQ3_EINVAL, "blob_read: section %d at %llu (+%llu), expected %llu (+%llu)", s,
                          (unsigned long long)h.offset[s], (unsigned long long)h.size[s],
                          (unsigned long long)want.offset[s], (unsigned long long)want.size[s]);
  if (h.total != want.total || bytes < h.total)
    return report_error(VQ3_EINVAL, "blob_read: %zu bytes, the blob needs %llu", bytes, (unsigned long long)want.total);
  if (fnv1a64(b + kHeaderBytes, h.total - kHeaderBytes) != h.hash)
    return report_error(VQ3_EINVAL, "blob_read: content hash mismatch (corrupt blob)");
  // the GPU-layout section must be the layout of the canonical stream
  std::vector<uint8_t> re(h.size[kPacked]);
  const int rc = vq3_pack_layout_fmt(h.format, b + h.offset[kCanon], h.d_in, h.d_out, re.data());
  if (rc) return rc;
  if (memcmp(re.data(), b + h.offset[kPacked], re.size()) != 0)
    return report_error(VQ3_EINVAL, "blob_read: the GPU-layout section is not the layout of the canonical stream");
  view->d_in = h.d_in;
  view->d_out = h.d_out;
  view->block = h.block;
  view->format = h.format;
  view->lr_rank = h.lr_rank;
  view->has_signs = (int)(h.flags & 1u);
  view->canonical = b + h.offset[kCanon];
  view->packed = b + h.offset[kPacked];
  view->scales = reinterpret_cast<const uint16_t*>(b + h.offset[kScales]);
  view->codebook = b + h.offset[kCodebook];
  view->codebook_bytes = h.size[kCodebook];
  view->signs = view->has_signs ? reinterpret_cast<const uint32_t*>(b + h.offset[kSigns]) : nullptr;
  view->lr_u = h.lr_rank ? reinterpret_cast<const uint16_t*>(b + h.offset[kU]) : nullptr;
  view->lr_v = h.lr_rank ? reinterpret_cast<const uint16_t*>(b + h.offset[kV]) : nullptr;
  return report_ok();
}

}  // extern "C"
