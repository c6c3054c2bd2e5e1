// C ABI of the VQ3 library: argument validation, host-side layout packing,
// workspace carving and kernel dispatch. No device memory is allocated here.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "vq3_internal.h"

namespace vq3 {
namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int ok() {
  g_err.clear();
  return VQ3_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(VQ3_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool pow2_block(int b) { return b >= 2 && b <= VQ3_MAX_BLOCK && (b & (b - 1)) == 0; }

int check_linear(const vq3_linear* L, const char* name) {
  if (!L) return fail(VQ3_EINVAL, "%s: null descriptor", name);
  if (L->d_in <= 0 || L->d_out <= 0) return fail(VQ3_EINVAL, "%s: d_in=%d d_out=%d must be positive", name, L->d_in, L->d_out);
  if (!layout_supported(L->d_in, L->d_out))
    return fail(VQ3_EUNSUPPORTED, "%s: d_in=%d must be a multiple of 64 and d_out=%d a multiple of 256", name, L->d_in,
                L->d_out);
  if (!pow2_block(L->block)) return fail(VQ3_EINVAL, "%s: block=%d must be a power of two in [2, 1024]", name, L->block);
  if (L->d_in % L->block) return fail(VQ3_EINVAL, "%s: d_in=%d is not a multiple of block=%d", name, L->d_in, L->block);
  if (!format_supported(L->format)) return fail(VQ3_EUNSUPPORTED, "%s: unknown index format %d", name, L->format);
  if (L->lr_rank < 0 || L->lr_rank > 64 || L->lr_rank % 8)
    return fail(VQ3_EUNSUPPORTED, "%s: lr_rank=%d must be 0 or a multiple of 8 up to 64", name, L->lr_rank);
  if (L->lr_rank && (!L->lr_u || !L->lr_v)) return fail(VQ3_EINVAL, "%s: null low-rank factors", name);
  if (L->lr_rank && (!aligned(L->lr_u, 16) || !aligned(L->lr_v, 16)))
    return fail(VQ3_EALIGN, "%s: low-rank factors must be 16-byte aligned", name);
  if (!L->packed || !L->codebook || !L->scales) return fail(VQ3_EINVAL, "%s: null packed/codebook/scales", name);
  if (!aligned(L->packed, 16)) return fail(VQ3_EALIGN, "%s: packed indices not 16-byte aligned", name);
  if (!aligned(L->codebook, 4) || !aligned(L->scales, 4) || (L->signs && !aligned(L->signs, 4)))
    return fail(VQ3_EALIGN, "%s: codebook, scales and signs must be 4-byte aligned", name);
  return VQ3_OK;
}

// ---- workspace carving ----------------------------------------------------

// Row tiles per pass of the persistent kernel for `rows` rows, passes of at
// most `pass_cap` rows (8, 16 or 32).
int pass_tiles(int rows, int pass_cap) { return dec_tiles_per_pass(rows < pass_cap ? rows : pass_cap); }

// Passes of the persistent kernel for `rows` rows.
int passes(int rows, int pass_cap) {
  const int per = 8 * pass_tiles(rows, pass_cap);
  return (rows + per - 1) / per;
}

// Pieces of one decode step of the persistent kernel.
size_t persist_pieces_bytes(int rows, int d_in, int d_out, int n_mats, int rank = 0) {
  const int nt = dec_tiles_per_pass(rows);
  const size_t piece = (size_t)512 * nt * sizeof(float);
  const size_t n_seg = (size_t)(d_out / kSuChannels) * n_mats;
  const int grid = persist_decode_grid(d_in, d_out, n_mats, persist_grid(nt));
  const int lw = rank ? persist_lowrank_weight(d_in, d_out, grid) : 0;
  return n_seg * persist_max_pieces(d_in, d_out, n_mats, grid, lw) * piece;
}

int seg_groups(int d_out, int n_mats) { return ((d_out / kSuChannels) * n_mats + kDecWarps - 1) / kDecWarps; }

// Counter words of the persistent kernel (word 0: finished CTAs).
struct CtlLayout {
  int off_g, off_hd, off_o, off_z, n;
};

CtlLayout ctl_mlp(int H, int I) {
  CtlLayout c{};
  c.off_g = 1;                          // gate/up segment groups
  c.off_hd = c.off_g + seg_groups(I, 2);  // h chunks (at most I/64): SwiGLU tasks done
  c.off_o = c.off_hd + I / 64;          // down segment groups
  c.n = c.off_o + seg_groups(H, 1);
  return c;
}

CtlLayout ctl_linear(int d_in, int d_out) {
  CtlLayout c{};
  c.off_o = c.off_g = c.off_hd = 1;
  c.off_z = c.off_o + seg_groups(d_out, 1);  // partials of the low-rank projection written
  c.n = c.off_z + 1;
  return c;
}

// Every workspace starts [status word (256 B)][counter words, zero between
// calls]. The decode kernel's hand-over counters and the prefill GEMM's part
// flags share the counter words, so one workspace serves any row count.
constexpr size_t kCtlOffset = 256;

size_t ctl_bytes(int n_words) {
  const int n = n_words > prefill_max_grid() ? n_words : prefill_max_grid();
  return round_up((size_t)n * sizeof(unsigned), 256);
}
size_t mlp_ctl_bytes(int H, int I) { return ctl_bytes(ctl_mlp(H, I).n); }
size_t linear_ctl_bytes(int d_in, int d_out) { return ctl_bytes(ctl_linear(d_in, d_out).n); }

// [status word][counter words][pieces]([partials of z = V x', one [8 * NT][64] FP32 per
// CTA of the first segment group] with low-rank factors)
struct LinearWs {
  size_t status, counters, pieces, lrz, total;
};

LinearWs linear_ws(int rows, int d_in, int d_out, int rank) {
  LinearWs w{};
  w.status = 0;
  w.counters = kCtlOffset;
  size_t off = kCtlOffset + linear_ctl_bytes(d_in, d_out);
  w.pieces = off;
  off = round_up(off + persist_pieces_bytes(rows, d_in, d_out, 1, rank), 256);
  w.lrz = off;
  if (rank) {
    const int nt = dec_tiles_per_pass(rows);
    const int grid = persist_decode_grid(d_in, d_out, 1, persist_grid(nt));
    const int lw = persist_lowrank_weight(d_in, d_out, grid);
    off = round_up(off + (size_t)persist_max_pieces(d_in, d_out, 1, grid, lw) * 512 * nt * sizeof(float), 256);
  }
  w.total = off;
  return w;
}

// [status word][counter words][h of one pass, fp32][gate/up pieces][down pieces]
struct MlpWs {
  size_t status, counters, hbuf, pieces1, pieces3, total;
};

MlpWs mlp_ws(int rows, const vq3_mlp_layer* l) {
  MlpWs w{};
  const int H = l->gate.d_in, I = l->gate.d_out;
  w.status = 0;
  w.counters = kCtlOffset;
  size_t off = kCtlOffset + mlp_ctl_bytes(H, I);
  w.hbuf = off;
  off = round_up(off + (size_t)8 * dec_tiles_per_pass(rows) * I * sizeof(float), 256);
  w.pieces1 = off;
  off = round_up(off + persist_pieces_bytes(rows, H, I, 2), 256);
  w.pieces3 = off;
  off = round_up(off + persist_pieces_bytes(rows, I, H, 1), 256);
  w.total = off;
  return w;
}

int check_mlp(const vq3_mlp_layer* l) {
  if (!l) return fail(VQ3_EINVAL, "mlp: null layer");
  int rc;
  if ((rc = check_linear(&l->gate, "gate"))) return rc;
  if ((rc = check_linear(&l->up, "up"))) return rc;
  if ((rc = check_linear(&l->down, "down"))) return rc;
  if (l->up.d_in != l->gate.d_in || l->up.d_out != l->gate.d_out || l->up.block != l->gate.block ||
      l->up.signs != l->gate.signs)
    return fail(VQ3_EINVAL, "mlp: gate and up must share d_in, d_out, block and signs");
  if (l->gate.lr_rank || l->up.lr_rank || l->down.lr_rank)
    return fail(VQ3_EUNSUPPORTED, "mlp: low-rank factors are supported on single linear layers only");
  if (l->up.format != l->gate.format || l->down.format != l->gate.format)
    return fail(VQ3_EINVAL, "mlp: gate, up and down must share one index format");
  if (l->down.d_in != l->gate.d_out || l->down.d_out != l->gate.d_in)
    return fail(VQ3_EINVAL, "mlp: down must be %d -> %d (got %d -> %d)", l->gate.d_out, l->gate.d_in, l->down.d_in,
                l->down.d_out);
  return VQ3_OK;
}

DecMat dec_mat(const vq3_linear& L) {
  DecMat m;
  m.packed = static_cast<const uint4*>(L.packed);
  m.codebook = reinterpret_cast<const uint32_t*>(L.codebook);
  m.scales = L.scales;
  return m;
}

// The persistent kernel over all rows, one launch per pass of 8/16/32 rows.
// `layer` null: a single linear layer L.
struct PersistBufs {
  float *hbuf, *pieces1, *pieces3;
  unsigned* ctl;
  int* status;
  float* lr_z;  // partials of z = V x' (linear layer with low-rank factors)
  // pre-norm residual step fused ahead of the MLP block (see PersistArgs::norm)
  int norm;
  const uint16_t* res_delta;
  uint16_t* res_out;
  float eps;
  const float* ss_in;  // residual stack chained by sums of squares (see PersistArgs)
  uint16_t* res_next;
  float* ss_next;
};

cudaError_t run_persistent(const uint16_t* x, int rows, int nt, const vq3_mlp_layer* layer, const vq3_linear* L,
                           const PersistBufs& b, uint16_t* out, cudaStream_t st) {
  PersistArgs a{};
  a.x = x;
  a.hbuf = b.hbuf;
  a.pieces1 = b.pieces1;
  a.pieces3 = b.pieces3;
  a.ctl = b.ctl;
  a.status = b.status;
  a.out = out;
  a.grid = persist_grid(nt);
  CtlLayout c{};
  if (layer) {
    const int H = layer->gate.d_in, I = layer->gate.d_out;
    a.mlp = 1;
    a.format = layer->gate.format;
    a.norm = b.norm;
    a.res_delta = b.res_delta;
    a.res_out = b.res_out;
    a.ss_in = b.ss_in;
    a.res_next = b.res_next;
    a.ss_next = b.ss_next;
    a.eps = b.eps;
    a.d_model = H;
    a.d_inter = I;
    a.d_model_out = H;
    a.block_in = layer->gate.block;
    a.signs_in = layer->gate.signs;
    a.block_dn = layer->down.block;
    a.signs_dn = layer->down.signs;
    a.x_chunk = persist_chunk(H, a.block_in);
    a.h_chunk = persist_chunk(I, a.block_dn);
    a.gate = dec_mat(layer->gate);
    a.up = dec_mat(layer->up);
    a.down = dec_mat(layer->down);
    a.grid1 = persist_decode_grid(H, I, 2, a.grid);
    a.max_pieces1 = persist_max_pieces(H, I, 2, a.grid1);
    a.grid3 = persist_decode_grid(I, H, 1, a.grid);
    a.max_pieces3 = persist_max_pieces(I, H, 1, a.grid3);
    c = ctl_mlp(H, I);
  } else {
    a.mlp = 0;
    a.format = L->format;
    if (L->lr_rank) {
      if (nt > 2) return cudaErrorInvalidValue;  // the projection's running sums cover up to 16 rows
      a.lr_v = L->lr_v;
      a.lr_u = L->lr_u;
      a.lr_rank = L->lr_rank;
      a.lr_z = b.lr_z;
    }
    a.d_model = L->d_in;
    a.d_model_out = L->d_out;
    a.block_in = L->block;
    a.signs_in = L->signs;
    a.x_chunk = persist_chunk(L->d_in, a.block_in);
    a.gate = a.up = a.down = dec_mat(*L);
    a.grid1 = persist_decode_grid(L->d_in, L->d_out, 1, a.grid);
    a.lr_lw = L->lr_rank ? persist_lowrank_weight(L->d_in, L->d_out, a.grid1) : 0;
    a.max_pieces1 = persist_max_pieces(L->d_in, L->d_out, 1, a.grid1, a.lr_lw);
    c = ctl_linear(L->d_in, L->d_out);
  }
  if (layer ? !(persist_cells_fit(a.d_model, a.d_inter, 2, a.grid1) && persist_cells_fit(a.d_inter, a.d_model, 1, a.grid3))
            : !persist_cells_fit(a.d_model, a.d_model_out, 1, a.grid1))
    return cudaErrorInvalidValue;
  a.scale_in = 1.0f / std::sqrt((float)a.block_in);
  a.scale_dn = a.mlp ? 1.0f / std::sqrt((float)a.block_dn) : 1.0f;
  a.n_ctl = c.n;
  a.off_g = c.off_g;
  a.off_hd = c.off_hd;
  a.off_o = c.off_o;
  a.off_z = c.off_z;
  for (int row0 = 0; row0 < rows; row0 += 8 * nt) {
    a.row0 = row0;
    a.rows = rows - row0 < 8 * nt ? rows - row0 : 8 * nt;
    cudaError_t e = launch_persistent(a, nt, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---- many-row (prefill) path: rotate, tensor-core GEMM with the LUT decoded
// into shared memory, (SwiGLU, rotate, GEMM)

constexpr int kPrefillRows = 17;  // from this many rows on, the tcgen05 path (the decode kernel is faster up to 16)

// [status word][counter words: part flags][x' FP16 [rows][d_in]]
// [h FP32 [rows][d_inter]][h' FP16 [rows][d_inter]][parts of split tiles]
// ([U V x' FP32 [rows][d_out]][projection parts FP32 [splits][rows][rank], then z [rows][rank]]
// with low-rank factors)
struct PrefillWs {
  size_t status, flags, xr, h, hr, part, ylr, zpart, total;
};

PrefillWs prefill_ws(int rows, int d_in, int d_inter, size_t ctl, int rank = 0, int d_out = 0) {
  PrefillWs w{};
  w.status = 0;
  w.flags = kCtlOffset;
  size_t off = kCtlOffset + ctl;
  w.xr = off;
  off = round_up(off + (size_t)rows * d_in * 2, 256);
  w.h = off;
  off = round_up(off + (size_t)rows * d_inter * 4, 256);
  w.hr = off;
  off = round_up(off + (size_t)rows * d_inter * 2, 256);
  w.part = off;
  off = round_up(off + prefill_part_bytes(rows), 256);
  w.ylr = w.zpart = off;
  if (rank) {
    off = round_up(off + (size_t)rows * d_out * sizeof(float), 256);
    w.zpart = off;
    off = round_up(off + lowrank_part_floats(d_in, rows, rank) * sizeof(float), 256);
  }
  w.total = off;
  return w;
}

PrefillArgs prefill_args(const uint16_t* xr, int rows, const vq3_linear& m0, const vq3_linear* m1, char* ws,
                         const PrefillWs& w) {
  PrefillArgs a{};
  a.x = xr;
  a.rows = rows;
  a.d_in = m0.d_in;
  a.d_out = m0.d_out;
  a.swiglu = m1 ? 1 : 0;
  a.format = m0.format;
  a.packed0 = static_cast<const uint4*>(m0.packed);
  a.cb0 = reinterpret_cast<const uint32_t*>(m0.codebook);
  a.scale0 = m0.scales;
  if (m1) {
    a.packed1 = static_cast<const uint4*>(m1->packed);
    a.cb1 = reinterpret_cast<const uint32_t*>(m1->codebook);
    a.scale1 = m1->scales;
  }
  a.status = reinterpret_cast<int*>(ws + w.status);
  a.flags = reinterpret_cast<unsigned*>(ws + w.flags);
  a.part = reinterpret_cast<float*>(ws + w.part);
  return a;
}

cudaError_t run_prefill_mlp(const uint16_t* x, int rows, const vq3_mlp_layer& l, char* ws, uint16_t* out,
                            cudaStream_t st) {
  const int H = l.gate.d_in, I = l.gate.d_out;
  const PrefillWs w = prefill_ws(rows, H, I, mlp_ctl_bytes(H, I));
  uint16_t* xr = reinterpret_cast<uint16_t*>(ws + w.xr);
  float* h = reinterpret_cast<float*>(ws + w.h);
  uint16_t* hr = reinterpret_cast<uint16_t*>(ws + w.hr);
  // x' and h' in the operand order of the GEMM kernel that serves this many rows
  const bool wide = prefill_wide(rows);
  auto gemm = wide ? launch_prefill_wide_gemm : launch_prefill_gemm;
  cudaError_t e = launch_fwht(x, rows, H, l.gate.block, l.gate.signs, xr, st, wide ? 0 : 1);
  if (e != cudaSuccess) return e;
  PrefillArgs gu = prefill_args(xr, rows, l.gate, &l.up, ws, w);
  gu.out32 = h;
  if ((e = gemm(gu, st)) != cudaSuccess) return e;
  if ((e = launch_fwht_f32(h, rows, I, l.down.block, l.down.signs, hr, st, wide ? 0 : 1)) != cudaSuccess) return e;
  PrefillArgs dn = prefill_args(hr, rows, l.down, nullptr, ws, w);
  dn.out16 = out;
  return gemm(dn, st);
}

cudaError_t run_prefill_linear(const uint16_t* x, int rows, const vq3_linear& L, char* ws, uint16_t* out,
                               cudaStream_t st) {
  const PrefillWs w = prefill_ws(rows, L.d_in, 0, linear_ctl_bytes(L.d_in, L.d_out), L.lr_rank, L.d_out);
  uint16_t* xr = reinterpret_cast<uint16_t*>(ws + w.xr);
  // x' in the operand order of the GEMM kernel that serves this many rows
  const bool wide = prefill_wide(rows);
  cudaError_t e = launch_fwht(x, rows, L.d_in, L.block, L.signs, xr, st, wide ? 0 : 1);
  if (e != cudaSuccess) return e;
  PrefillArgs a = prefill_args(xr, rows, L, nullptr, ws, w);
  if (L.lr_rank) {
    float* ylr = reinterpret_cast<float*>(ws + w.ylr);
    float* zpart = reinterpret_cast<float*>(ws + w.zpart);
    if ((e = launch_lowrank(xr, rows, L.d_in, L.lr_v, L.lr_u, L.lr_rank, L.d_out, zpart, ylr, st, wide ? 0 : 1)) !=
        cudaSuccess)
      return e;
    a.lr_y = ylr;
  }
  a.out16 = out;
  return wide ? launch_prefill_wide_gemm(a, st) : launch_prefill_gemm(a, st);
}

// Runs fn(i) for i in [0, n) on up to hardware_concurrency host threads (the
// channel groups of a matrix touch disjoint bytes of both layouts).
template <typename F>
void parallel_for(int n, F fn) {
  unsigned hw = std::thread::hardware_concurrency();
  const int nt = (int)(hw == 0 ? 1 : (hw > 64 ? 64 : hw));
  const int k = n < nt ? n : nt;
  if (k <= 1) {
    for (int i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> th;
  th.reserve(k);
  for (int j = 0; j < k; ++j)
    th.emplace_back([=] {
      for (int i = j; i < n; i += k) fn(i);
    });
  for (auto& x : th) x.join();
}

// Index k of a canonical stream of nb-bit indices (nb = 4 or 6).
uint32_t read_index(const uint8_t* s, size_t k, int nb) {
  const size_t bit = (size_t)nb * k;
  const size_t byte = bit / 8;
  const unsigned sh = (unsigned)(bit % 8);
  uint32_t v = s[byte];
  if (sh + nb > 8) v |= (uint32_t)s[byte + 1] << 8;
  return (v >> sh) & ((1u << nb) - 1u);
}

// Where index n of lane `lane`'s string in SU (mg, kg) belongs: its canonical
// output group (pair for the vector formats, channel for the scalar one) and input.
struct LanePos {
  int group, input;
};
LanePos lane_pos(int format, int mg, int kg, int lane, int n) {
  static const int koff[4] = {0, 1, 8, 9};
  const int g = lane / 4, t = lane % 4;
  const int c = format_vec(format) == 1 ? n % 2 : 0;
  const int nn = format_vec(format) == 1 ? n / 2 : n;
  const int s = nn / 16, m = (nn / 4) % 4, e = nn % 4;
  const int p = mg * 32 + m * 8 + g;
  LanePos q;
  q.group = format_vec(format) == 1 ? 2 * p + c : p;
  q.input = kg * 64 + s * 16 + 2 * t + koff[e];
  return q;
}

}  // namespace

int mlp_validate(const uint16_t* x, int rows, const vq3_mlp_layer* layer, const uint16_t* out) {
  int rc = check_mlp(layer);
  if (rc) return rc;
  if (rows < 0) return fail(VQ3_EINVAL, "mlp: rows=%d", rows);
  if (rows == 0) return VQ3_OK;
  if (!x || !out) return fail(VQ3_EINVAL, "mlp: null x/out");
  if (!aligned(x, 16) || !aligned(out, 16)) return fail(VQ3_EALIGN, "mlp: x/out must be 16-byte aligned");
  return VQ3_OK;
}

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;  // no device visible: size for a GB300
  }
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

void mlp_counter_range(const vq3_mlp_layer* layer, size_t* offset, size_t* bytes) {
  *offset = kCtlOffset;
  *bytes = mlp_ctl_bytes(layer->gate.d_in, layer->gate.d_out);
}

// For the other host-side files of the library: the same thread-local error message.
int report_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}
int report_ok() { return ok(); }

}  // namespace vq3

using namespace vq3;

extern "C" {

const char* vq3_last_error(void) { return g_err.c_str(); }

const char* vq3_version(void) {
#ifdef VQ3_BOUNDS_CHECK
  return "vq3-gb300 0.2 (sm_103a; layout su64x64-m16n8k16; bounds-check build)";
#else
  return "vq3-gb300 0.2 (sm_103a; layout su64x64-m16n8k16)";
#endif
}

int vq3_bounds_check(unsigned* out, int n_out, int reset) {
#ifdef VQ3_BOUNDS_CHECK
  if (!out || n_out < 2 * VQ3_BOUNDS_FILES)
    return report_error(VQ3_EINVAL, "bounds_check: out needs %d entries", 2 * VQ3_BOUNDS_FILES);
  cudaError_t (*const rd[VQ3_BOUNDS_FILES])(unsigned*, bool) = {bounds_read_persistent, bounds_read_lowrank,
                                                                 bounds_read_delta,      bounds_read_rotate,
                                                                 bounds_read_prefill,    bounds_read_prefill_wide};
  for (int f = 0; f < VQ3_BOUNDS_FILES; ++f) {
    const cudaError_t e = rd[f](out + 2 * f, reset != 0);
    if (e != cudaSuccess) return report_error(VQ3_ECUDA, "bounds_check: %s", cudaGetErrorString(e));
  }
  return report_ok();
#else
  (void)out;
  (void)n_out;
  (void)reset;
  return report_error(VQ3_EUNSUPPORTED, "bounds_check: this library was built without -DVQ3_BOUNDS_CHECK");
#endif
}

size_t vq3_packed_bytes_fmt(int format, int d_in, int d_out) {
  if (!format_supported(format) || !layout_supported(d_in, d_out)) return 0;
  return (size_t)(d_out / kSuChannels) * (size_t)(d_in / kSuInputs) * (size_t)format_su_bytes(format);
}

size_t vq3_packed_bytes(int d_in, int d_out) { return vq3_packed_bytes_fmt(VQ3_FORMAT_2X64, d_in, d_out); }

int vq3_pack_layout_fmt(int format, const uint8_t* canonical, int d_in, int d_out, void* dst_host) {
  if (!canonical || !dst_host) return fail(VQ3_EINVAL, "pack_layout: null pointer");
  if (!format_supported(format)) return fail(VQ3_EUNSUPPORTED, "pack_layout: unknown format %d", format);
  if (!layout_supported(d_in, d_out))
    return fail(VQ3_EUNSUPPORTED, "pack_layout: d_in=%d and d_out=%d must be positive multiples of 64", d_in, d_out);
  uint8_t* dst = static_cast<uint8_t*>(dst_host);
  const int n_mg = d_out / kSuChannels, n_kg = d_in / kSuInputs;
  const int nb = format_bits(format), vec = format_vec(format), words = format_words(format);
  const int su_bytes = format_su_bytes(format), n_idx = 128 / vec;
  parallel_for(n_mg, [=](int mg) {
    for (int kg = 0; kg < n_kg; ++kg) {
      const size_t su = (size_t)mg * n_kg + kg;
      for (int lane = 0; lane < 32; ++lane) {
        uint32_t w[17] = {0};
        for (int n = 0; n < n_idx; ++n) {
          const LanePos q = lane_pos(format, mg, kg, lane, n);
          const uint32_t idx = read_index(canonical, (size_t)q.group * d_in + q.input, nb);
          const int bit = nb * n;
          w[bit / 32] |= idx << (bit % 32);
          if (bit % 32 + nb > 32) w[bit / 32 + 1] |= idx >> (32 - bit % 32);
        }
        for (int wi = 0; wi < words; ++wi) memcpy(dst + lane_word_offset(su, lane, wi, su_bytes), &w[wi], 4);
      }
    }
  });
  return ok();
}

int vq3_pack_layout(const uint8_t* canonical, int d_in, int d_out, void* dst_host) {
  return vq3_pack_layout_fmt(VQ3_FORMAT_2X64, canonical, d_in, d_out, dst_host);
}

int vq3_unpack_layout_fmt(int format, const void* packed_host, int d_in, int d_out, uint8_t* canonical) {
  if (!canonical || !packed_host) return fail(VQ3_EINVAL, "unpack_layout: null pointer");
  if (!format_supported(format)) return fail(VQ3_EUNSUPPORTED, "unpack_layout: unknown format %d", format);
  if (!layout_supported(d_in, d_out))
    return fail(VQ3_EUNSUPPORTED, "unpack_layout: d_in=%d and d_out=%d must be positive multiples of 64", d_in, d_out);
  const uint8_t* src = static_cast<const uint8_t*>(packed_host);
  const int nb = format_bits(format), vec = format_vec(format), words = format_words(format);
  const int su_bytes = format_su_bytes(format), n_idx = 128 / vec;
  const size_t count = (size_t)(d_out / vec) * d_in;
  memset(canonical, 0, (nb * count + 7) / 8);
  const int n_mg = d_out / kSuChannels, n_kg = d_in / kSuInputs;
  parallel_for(n_mg, [=](int mg) {
    for (int kg = 0; kg < n_kg; ++kg) {
      const size_t su = (size_t)mg * n_kg + kg;
      for (int lane = 0; lane < 32; ++lane) {
        uint32_t w[17] = {0};
        for (int wi = 0; wi < words; ++wi) memcpy(&w[wi], src + lane_word_offset(su, lane, wi, su_bytes), 4);
        for (int n = 0; n < n_idx; ++n) {
          const LanePos q = lane_pos(format, mg, kg, lane, n);
          const int bit = nb * n;
          const uint64_t v = ((uint64_t)w[bit / 32 + 1] << 32) | w[bit / 32];
          const uint32_t idx = (uint32_t)(v >> (bit % 32)) & ((1u << nb) - 1u);
          // one channel group mg spans a whole number of stream bytes (64 channels x
          // d_in inputs, d_in a multiple of 64), so threads on different mg never
          // write the same byte
          const size_t sb = (size_t)nb * ((size_t)q.group * d_in + q.input);
          canonical[sb / 8] |= (uint8_t)(idx << (sb % 8));
          if (sb % 8 + nb > 8) canonical[sb / 8 + 1] |= (uint8_t)(idx >> (8 - sb % 8));
        }
      }
    }
  });
  return ok();
}

int vq3_unpack_layout(const void* packed_host, int d_in, int d_out, uint8_t* canonical) {
  return vq3_unpack_layout_fmt(VQ3_FORMAT_2X64, packed_host, d_in, d_out, canonical);
}

int fwht_rotate(const uint16_t* x, int rows, int n, int block, const uint32_t* signs, uint16_t* out, void* stream) {
  if (rows < 0 || n <= 0) return fail(VQ3_EINVAL, "fwht_rotate: rows=%d n=%d", rows, n);
  if (!pow2_block(block)) return fail(VQ3_EINVAL, "fwht_rotate: block=%d must be a power of two in [2, 1024]", block);
  if (n % block) return fail(VQ3_EINVAL, "fwht_rotate: n=%d is not a multiple of block=%d", n, block);
  if (rows == 0) return ok();
  if (!x || !out) return fail(VQ3_EINVAL, "fwht_rotate: null x/out");
  if (!aligned(x, 16) || !aligned(out, 16) || (signs && !aligned(signs, 4)))
    return fail(VQ3_EALIGN, "fwht_rotate: x/out must be 16-byte aligned, signs 4-byte aligned");
  cudaError_t e = launch_fwht(x, rows, n, block, signs, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fwht_rotate launch");
  return ok();
}

size_t vq3_linear_workspace_bytes(int rows, const vq3_linear* L) {
  if (!L || rows < 0 || !layout_supported(L->d_in, L->d_out)) return 0;
  if (rows >= kPrefillRows)
    return prefill_ws(rows, L->d_in, 0, linear_ctl_bytes(L->d_in, L->d_out), L->lr_rank, L->d_out).total;
  return linear_ws(rows, L->d_in, L->d_out, L->lr_rank).total;
}

size_t vq3_mlp_workspace_bytes(int rows, const vq3_mlp_layer* layer) {
  if (!layer || rows < 0 || !layout_supported(layer->gate.d_in, layer->gate.d_out)) return 0;
  const int H = layer->gate.d_in, I = layer->gate.d_out;
  if (rows >= kPrefillRows) return prefill_ws(rows, H, I, mlp_ctl_bytes(H, I)).total;
  return mlp_ws(rows, layer).total;
}

int vq3_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace) return fail(VQ3_EINVAL, "workspace_init: null workspace");
  cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace_init memset");
  return ok();
}

int vq3_workspace_status(const void* workspace, int* status_host, void* stream) {
  if (!workspace || !status_host) return fail(VQ3_EINVAL, "workspace_status: null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(status_host, workspace, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "workspace_status copy");
  return ok();
}

int vq3_linear_forward(const uint16_t* x, int rows, const vq3_linear* L, uint16_t* out, void* workspace,
                       size_t ws_bytes, void* stream) {
  int rc = check_linear(L, "linear");
  if (rc) return rc;
  if (rows < 0) return fail(VQ3_EINVAL, "linear: rows=%d", rows);
  if (rows == 0) return ok();
  if (!x || !out || !workspace) return fail(VQ3_EINVAL, "linear: null x/out/workspace");
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(workspace, 256))
    return fail(VQ3_EALIGN, "linear: x/out must be 16-byte aligned and the workspace 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if (rows >= kPrefillRows) {
    const size_t need = prefill_ws(rows, L->d_in, 0, linear_ctl_bytes(L->d_in, L->d_out), L->lr_rank, L->d_out).total;
    if (ws_bytes < need) return fail(VQ3_ENOSPACE, "linear: workspace %zu < %zu bytes", ws_bytes, need);
    cudaError_t e = run_prefill_linear(x, rows, *L, ws, out, st);
    if (e != cudaSuccess) return cuda_fail(e, "linear: launch");
    return ok();
  }
  const LinearWs w = linear_ws(rows, L->d_in, L->d_out, L->lr_rank);
  if (ws_bytes < w.total) return fail(VQ3_ENOSPACE, "linear: workspace %zu < %zu bytes", ws_bytes, w.total);
  PersistBufs b{};
  b.pieces1 = reinterpret_cast<float*>(ws + w.pieces);
  b.ctl = reinterpret_cast<unsigned*>(ws + w.counters);
  b.status = reinterpret_cast<int*>(ws + w.status);
  b.lr_z = reinterpret_cast<float*>(ws + w.lrz);  // the low-rank correction is formed inside the kernel
  cudaError_t e = run_persistent(x, rows, dec_tiles_per_pass(rows), nullptr, L, b, out, st);
  if (e != cudaSuccess) return cuda_fail(e, "linear: launch");
  return ok();
}

namespace {

struct MlpCall {
  int rc;
  MlpWs w;
  char* ws;
  cudaStream_t st;
};

MlpCall mlp_prepare(int rows, int pass_cap, const vq3_mlp_layer* layer, void* workspace, size_t ws_bytes,
                    void* stream, const char* name) {
  MlpCall c{};
  c.rc = check_mlp(layer);
  if (c.rc) return c;
  if (rows < 0) {
    c.rc = fail(VQ3_EINVAL, "%s: rows=%d", name, rows);
    return c;
  }
  if (rows == 0) return c;
  if (!workspace) {
    c.rc = fail(VQ3_EINVAL, "%s: null workspace", name);
    return c;
  }
  if (!aligned(workspace, 256)) {
    c.rc = fail(VQ3_EALIGN, "%s: workspace must be 256-byte aligned", name);
    return c;
  }
  c.w = mlp_ws(rows < pass_cap ? rows : pass_cap, layer);
  if (ws_bytes < c.w.total) {
    c.rc = fail(VQ3_ENOSPACE, "%s: workspace %zu < %zu bytes", name, ws_bytes, c.w.total);
    return c;
  }
  c.ws = static_cast<char*>(workspace);
  c.st = static_cast<cudaStream_t>(stream);
  return c;
}

}  // namespace

}  // extern "C"

namespace vq3 {

size_t mlp_workspace_bytes_capped(int rows, const vq3_mlp_layer* layer, int pass_cap) {
  if (!layer || rows < 0 || !layout_supported(layer->gate.d_in, layer->gate.d_out)) return 0;
  return mlp_ws(rows < pass_cap ? rows : pass_cap, layer).total;
}

namespace {
// The decode-kernel MLP path; `norm` (optional) carries the fused pre-norm residual step.
int mlp_forward_decode(const uint16_t* x, int rows, const vq3_mlp_layer* layer, uint16_t* out, void* workspace,
                       size_t ws_bytes, void* stream, int pass_cap, const PersistBufs* norm) {
  MlpCall c = mlp_prepare(rows, pass_cap, layer, workspace, ws_bytes, stream, "mlp");
  if (c.rc || rows == 0) return c.rc ? c.rc : ok();
  if (!x || !out) return fail(VQ3_EINVAL, "mlp: null x/out");
  if (!aligned(x, 16) || !aligned(out, 16)) return fail(VQ3_EALIGN, "mlp: x/out must be 16-byte aligned");
  PersistBufs b{};
  if (norm) {
    b.norm = 1;
    b.res_delta = norm->res_delta;
    b.res_out = norm->res_out;
    b.eps = norm->eps;
    b.ss_in = norm->ss_in;
    b.res_next = norm->res_next;
    b.ss_next = norm->ss_next;
  }
  b.hbuf = reinterpret_cast<float*>(c.ws + c.w.hbuf);
  b.pieces1 = reinterpret_cast<float*>(c.ws + c.w.pieces1);
  b.pieces3 = reinterpret_cast<float*>(c.ws + c.w.pieces3);
  b.ctl = reinterpret_cast<unsigned*>(c.ws + c.w.counters);
  b.status = reinterpret_cast<int*>(c.ws + c.w.status);
  cudaError_t e = run_persistent(x, rows, pass_tiles(rows, pass_cap), layer, nullptr, b, out, c.st);
  if (e != cudaSuccess) return cuda_fail(e, "mlp: launch");
  return ok();
}
}  // namespace

int mlp_forward_capped(const uint16_t* x, int rows, const vq3_mlp_layer* layer, uint16_t* out, void* workspace,
                       size_t ws_bytes, void* stream, int pass_cap) {
  return mlp_forward_decode(x, rows, layer, out, workspace, ws_bytes, stream, pass_cap, nullptr);
}

}  // namespace vq3

extern "C" {

int vq3_mlp_forward(const uint16_t* x, int rows, const vq3_mlp_layer* layer, uint16_t* out, void* workspace,
                    size_t ws_bytes, void* stream) {
  if (rows < kPrefillRows) return mlp_forward_capped(x, rows, layer, out, workspace, ws_bytes, stream, 32);
  int rc = check_mlp(layer);
  if (rc) return rc;
  if (!x || !out || !workspace) return fail(VQ3_EINVAL, "mlp: null x/out/workspace");
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(workspace, 256))
    return fail(VQ3_EALIGN, "mlp: x/out must be 16-byte aligned and the workspace 256-byte aligned");
  const int H = layer->gate.d_in, I = layer->gate.d_out;
  const size_t need = prefill_ws(rows, H, I, mlp_ctl_bytes(H, I)).total;
  if (ws_bytes < need) return fail(VQ3_ENOSPACE, "mlp: workspace %zu < %zu bytes", ws_bytes, need);
  cudaError_t e = run_prefill_mlp(x, rows, *layer, static_cast<char*>(workspace), out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mlp: launch");
  return ok();
}

int vq3_delta_rule_forward(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* beta,
                           const float* alpha, int tokens, int heads, int d_k, int d_v, float* state, uint16_t* out,
                           void* stream) {
  if (tokens < 0 || heads <= 0) return fail(VQ3_EINVAL, "delta_rule: tokens=%d heads=%d", tokens, heads);
  if (d_k < 8 || d_k > 256 || d_k % 8 || d_v <= 0 || d_v % 16)
    return fail(VQ3_EUNSUPPORTED, "delta_rule: d_k=%d must be a multiple of 8 in [8, 256], d_v=%d a multiple of 16",
                d_k, d_v);
  if (!state) return fail(VQ3_EINVAL, "delta_rule: null state");
  if (tokens == 0) return ok();
  if (!q || !k || !v || !beta || !alpha || !out) return fail(VQ3_EINVAL, "delta_rule: null pointer");
  cudaError_t e = launch_delta_rule(q, k, v, beta, alpha, tokens, heads, d_k, d_v, state, out,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "delta_rule: launch");
  return ok();
}

int vq3_mlp_forward_residual(const uint16_t* r_in, const uint16_t* delta, int rows, const vq3_mlp_layer* layer,
                             float eps, uint16_t* r_out, uint16_t* out, void* workspace, size_t ws_bytes,
                             void* stream) {
  if (rows < 0 || !(eps >= 0.f)) return fail(VQ3_EINVAL, "mlp_residual: rows=%d eps=%g", rows, eps);
  int rc = check_mlp(layer);
  if (rc) return rc;
  if (rows == 0) return ok();
  if (!r_in || !r_out || !out || !workspace) return fail(VQ3_EINVAL, "mlp_residual: null pointer");
  if (r_out == r_in || (delta && r_out == delta) || out == r_in || out == r_out || (delta && out == delta))
    return fail(VQ3_EINVAL, "mlp_residual: r_out and out must not alias r_in, delta or each other");
  if (!aligned(r_in, 16) || !aligned(r_out, 16) || !aligned(out, 16) || (delta && !aligned(delta, 16)))
    return fail(VQ3_EALIGN, "mlp_residual: pointers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows < kPrefillRows) {
    PersistBufs nb{};
    nb.res_delta = delta;
    nb.res_out = r_out;
    nb.eps = eps;
    return mlp_forward_decode(r_in, rows, layer, out, workspace, ws_bytes, stream, 32, &nb);
  }
  // many rows: the RMSNorm kernel writes r' and the normed rows (into out, which the block
  // reads before it writes its result there), then the tensor-core path
  const int H = layer->gate.d_in, I = layer->gate.d_out;
  const size_t need = prefill_ws(rows, H, I, mlp_ctl_bytes(H, I)).total;
  if (ws_bytes < need) return fail(VQ3_ENOSPACE, "mlp_residual: workspace %zu < %zu bytes", ws_bytes, need);
  cudaError_t e = launch_residual_rmsnorm2(r_in, delta, r_out, rows, H, eps, out, st);
  if (e == cudaSuccess) e = run_prefill_mlp(out, rows, *layer, static_cast<char*>(workspace), out, st);
  if (e != cudaSuccess) return cuda_fail(e, "mlp_residual: launch");
  return ok();
}

int vq3_mlp_prenorm_step(const uint16_t* r, const float* ss, int rows, const vq3_mlp_layer* layer, float eps,
                         uint16_t* out, uint16_t* r_next, float* ss_next, void* workspace, size_t ws_bytes,
                         void* stream) {
  if (rows < 0 || !(eps >= 0.f)) return fail(VQ3_EINVAL, "mlp_prenorm: rows=%d eps=%g", rows, eps);
  int rc = check_mlp(layer);
  if (rc) return rc;
  if (rows == 0) return ok();
  if (!r || !out || !r_next || !workspace) return fail(VQ3_EINVAL, "mlp_prenorm: null pointer");
  if (out == r || r_next == r || r_next == out || (ss && ss_next && (const void*)ss == (const void*)ss_next))
    return fail(VQ3_EINVAL, "mlp_prenorm: out, r_next and ss_next must not alias r, ss or each other");
  if (!aligned(r, 16) || !aligned(out, 16) || !aligned(r_next, 16) || (ss && !aligned(ss, 16)) ||
      (ss_next && !aligned(ss_next, 16)))
    return fail(VQ3_EALIGN, "mlp_prenorm: pointers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows < kPrefillRows) {
    PersistBufs nb{};
    nb.eps = eps;
    nb.ss_in = ss;
    nb.res_next = r_next;
    nb.ss_next = ss_next;
    return mlp_forward_decode(r, rows, layer, out, workspace, ws_bytes, stream, 32, &nb);
  }
  // many rows: the RMSNorm kernel writes the normed rows into out (the block reads them
  // before it writes its result there), the tensor-core path, then the residual step
  const int H = layer->gate.d_in, I = layer->gate.d_out;
  const size_t need = prefill_ws(rows, H, I, mlp_ctl_bytes(H, I)).total;
  if (ws_bytes < need) return fail(VQ3_ENOSPACE, "mlp_prenorm: workspace %zu < %zu bytes", ws_bytes, need);
  cudaError_t e = launch_residual_rmsnorm2(r, nullptr, const_cast<uint16_t*>(r), rows, H, eps, out, st);
  if (e == cudaSuccess) e = run_prefill_mlp(out, rows, *layer, static_cast<char*>(workspace), out, st);
  if (e == cudaSuccess) e = launch_residual_add_ss(r, out, r_next, ss_next, rows, H, st);
  if (e != cudaSuccess) return cuda_fail(e, "mlp_prenorm: launch");
  return ok();
}

int vq3_mlp_kernel_launches(int rows, const vq3_mlp_layer* layer) {
  if (check_mlp(layer) || rows < 0) return -1;
  if (rows == 0) return 0;
  if (rows >= kPrefillRows) return 4;  // rotate x, gate/up GEMM, rotate h, down GEMM
  return passes(rows, 32);             // one persistent kernel per pass of 8, 16 or 32 rows
}

int vq3_linear_kernel_launches(int rows, const vq3_linear* L) {
  if (check_linear(L, "linear") || rows < 0) return -1;
  if (rows == 0) return 0;
  if (rows >= kPrefillRows) return L->lr_rank ? 5 : 2;  // rotate x, (project, reduce, expand,) GEMM
  return 1;  // the decode kernel alone, the low-rank correction formed inside it
}

size_t vq3_mlp_host_workspace_bytes(int rows, const vq3_mlp_layer* layer) {
  const size_t base = vq3_mlp_workspace_bytes(rows, layer);
  if (!base) return 0;
  const size_t io = round_up((size_t)rows * layer->gate.d_in * 2, 256);
  return base + 2 * io;
}

int vq3_mlp_forward_host(const uint16_t* x_host, int rows, const vq3_mlp_layer* layer, uint16_t* out_host,
                         void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_mlp(layer);
  if (rc) return rc;
  if (rows < 0) return fail(VQ3_EINVAL, "mlp_host: rows=%d", rows);
  if (rows == 0) return ok();
  if (!x_host || !out_host || !workspace) return fail(VQ3_EINVAL, "mlp_host: null x/out/workspace");
  if (!aligned(workspace, 256)) return fail(VQ3_EALIGN, "mlp_host: workspace must be 256-byte aligned");
  const size_t need = vq3_mlp_host_workspace_bytes(rows, layer);
  if (ws_bytes < need) return fail(VQ3_ENOSPACE, "mlp_host: workspace %zu < %zu bytes", ws_bytes, need);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)rows * layer->gate.d_in * 2;
  const size_t io = round_up(bytes, 256);
  char* ws = static_cast<char*>(workspace);
  uint16_t* xd = reinterpret_cast<uint16_t*>(ws);
  uint16_t* yd = reinterpret_cast<uint16_t*>(ws + io);
  cudaError_t e = cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "mlp_host: copy in");
  rc = vq3_mlp_forward(xd, rows, layer, yd, ws + 2 * io, ws_bytes - 2 * io, stream);
  if (rc) return rc;
  e = cudaMemcpyAsync(out_host, yd, bytes, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "mlp_host: copy out");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "mlp_host: synchronize");
  return ok();
}

int vq3_residual_rmsnorm(uint16_t* resid, const uint16_t* delta, int rows, int n, float eps, uint16_t* normed,
                         void* stream) {
  if (rows < 0 || n <= 0 || !(eps >= 0.f)) return fail(VQ3_EINVAL, "residual_rmsnorm: rows=%d n=%d eps=%g", rows, n, eps);
  if (rows == 0) return ok();
  if (!resid || !normed) return fail(VQ3_EINVAL, "residual_rmsnorm: null resid/normed");
  if (!aligned(resid, 16) || !aligned(normed, 16) || (delta && !aligned(delta, 16)))
    return fail(VQ3_EALIGN, "residual_rmsnorm: pointers must be 16-byte aligned");
  cudaError_t e = launch_residual_rmsnorm(resid, delta, rows, n, eps, normed, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "residual_rmsnorm launch");
  return ok();
}

int vq3_dequant_dense(const vq3_linear* L, int apply_scale, uint16_t* w_out, void* stream) {
  int rc = check_linear(L, "dequant");
  if (rc) return rc;
  if (!w_out) return fail(VQ3_EINVAL, "dequant: null w_out");
  if (!aligned(w_out, 16)) return fail(VQ3_EALIGN, "dequant: w_out must be 16-byte aligned");
  cudaError_t e = launch_dequant(*L, apply_scale ? 1 : 0, w_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
  return ok();
}

}  // extern "C"
