/*
 * vq3.h - C ABI of the VQ3 Hadamard-rotated vector-LUT MLP library (sm_103a).
 *
 * What the library computes (page titles and sections of the sources):
 *   model card "anemll/anemll-forge-qwen3.8-27B", section "Release 0.2:
 *   three-bit MLP, token-mixer rotations, distilled weights":
 *     - every MLP matrix (gate, up, down) is a three-bit vector lookup table
 *       "2x64": a codebook of 64 two-component FP16 centroids per matrix, one
 *       six-bit index per pair of output channels (per input column), and an
 *       FP16 scale per output channel;
 *     - the input of each matrix is multiplied online by 1,024-wide Hadamard
 *       blocks with seeded signs, the weights being stored in the rotated basis.
 *   "ANEMLL ANE LLM conversion pipeline", section "Facts": the SiLU of the
 *   gated MLP is 0.5*x*(1+tanh(x/2)) = x*sigmoid(x); vector LUTs run along
 *   output channels.
 *
 * So for one matrix with d_out outputs and d_in inputs:
 *   x'      = blockdiag(H_b diag(s)) x / sqrt(b)           (per row, b = block)
 *   W[2p+c][i] = scale[2p+c] * C[idx[p][i]][c]             (c in {0,1})
 *   y       = W x'
 * and an MLP block is y = W_d R_d( silu(W_g R x) * (W_u R x) ).
 *
 * Conventions (every entry point):
 *   - Return value: VQ3_OK (0) or a negative VQ3_E* code; vq3_last_error()
 *     then returns a thread-local message. No C++ exception crosses the ABI.
 *   - The caller owns every buffer. Activation, output and packed-index
 *     pointers must be 16-byte aligned, codebook, scale and sign pointers
 *     4-byte aligned and workspaces 256-byte aligned (VQ3_EALIGN otherwise).
 *     The library never allocates device memory; the entry points that need
 *     scratch take a caller-supplied workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Device work is enqueued asynchronously on it; arguments are
 *     validated on the host before anything is enqueued, so an error return
 *     means nothing was launched.
 *   - FP16 data is passed as uint16_t bit patterns (IEEE binary16).
 *   - Activations are row-major [rows][n]; rows == 0 is a valid no-op.
 */
#ifndef VQ3_H_
#define VQ3_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VQ3_API __attribute__((visibility("default")))
#else
#define VQ3_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define VQ3_OK 0
#define VQ3_EINVAL (-1)       /* bad size, null pointer or inconsistent descriptor */
#define VQ3_EALIGN (-2)       /* a pointer breaks the alignment rule above */
#define VQ3_EUNSUPPORTED (-3) /* shape outside what the kernels implement */
#define VQ3_ECUDA (-4)        /* a CUDA runtime call failed (message has the CUDA error) */
#define VQ3_ENOSPACE (-5)     /* workspace smaller than the size query returned */

#define VQ3_CODEBOOK_SIZE 64
#define VQ3_MAX_BLOCK 1024

/*
 * Index formats (vq3_linear.format). Cited: model card
 * "anemll/anemll-forge-qwen3.8-27B", "Release 0.2" bullet "Three bits per MLP
 * weight" (2x64) and the release-comparison table rows "MLP gate / up / down"
 * and "Token mixers" (the previous release's two-bit vector LUT, 2x16, and
 * four-bit LUT). Every format has per-output-channel FP16 scales.
 *   VQ3_FORMAT_2X64: 64 two-component FP16 centroids, one 6-bit index per
 *                    output pair and input (3 bits per weight).
 *   VQ3_FORMAT_2X16: 16 two-component FP16 centroids, one 4-bit index per
 *                    output pair and input (2 bits per weight).
 *   VQ3_FORMAT_LUT4: 16 scalar FP16 entries, one 4-bit index per weight
 *                    (4 bits per weight).
 * Canonical stream of a format with index width b and v output channels per
 * index: index k = p*d_in + i (output group p = channels v*p .. v*p+v-1, input
 * column i) occupies stream bits [b*k, b*k + b), stream bit j being bit (j mod 8)
 * of byte j/8 (least significant bit first); ceil(b*(d_out/v)*d_in/8) bytes.
 */
#define VQ3_FORMAT_2X64 0
#define VQ3_FORMAT_2X16 1
#define VQ3_FORMAT_LUT4 2

/*
 * One VQ3 matrix, d_out x d_in. Cited: model card "anemll/anemll-forge-qwen3.8-27B",
 * "Release 0.2" bullet "Three bits per MLP weight" (and the formats above).
 *   d_in  : input width; a multiple of 64 and of `block`.
 *   d_out : output width; a multiple of 64 (so output channels pair up).
 *   block : Hadamard block of the input rotation, a power of two in [2, 1024].
 *   packed: device, 16-byte aligned, vq3_packed_bytes_fmt(format, d_in, d_out)
 *           bytes in the GPU layout written by vq3_pack_layout_fmt.
 *   codebook: device, FP16 centroids: [64][2] (2X64), [16][2] (2X16; component
 *           0 = even channel of the pair) or [16] (LUT4); 4-byte aligned.
 *   scales: device, [d_out] FP16 per-output-channel scales.
 *   signs : device, bit-packed seeded signs over d_in (bit j of word j/32 set
 *           => input j is negated before the Hadamard block), or NULL for all +1.
 *   format: VQ3_FORMAT_*.
 *   lr_rank, lr_u, lr_v: optional low-rank correction (model card
 *           "anemll/anemll-forge-qwen3.8-27B", table row "Token mixers": rank-64
 *           factors): the weight becomes diag(scales) C[idx] + U V, with U =
 *           lr_u [d_out][lr_rank] and V = lr_v [lr_rank][d_in], device FP16,
 *           16-byte aligned, acting on the rotated input like the lookup-table
 *           part (the scales apply to the lookup-table part only). lr_rank = 0
 *           (no factors) or a multiple of 8 up to 64. Single linear layers only:
 *           vq3_mlp_forward rejects matrices with factors.
 */
typedef struct vq3_linear {
  int d_in;
  int d_out;
  int block;
  const void* packed;
  const uint16_t* codebook;
  const uint16_t* scales;
  const uint32_t* signs;
  int format;  // VQ3_FORMAT_*; 0 (the three-bit format) in a zero-initialised descriptor
  int lr_rank;  // 0: no low-rank correction
  const uint16_t* lr_u;
  const uint16_t* lr_v;
} vq3_linear;

/* One SwiGLU block. gate and up read the same rotated input (same d_in, block
 * and signs); down maps the intermediate width back: down.d_in == gate.d_out,
 * down.d_out == gate.d_in. The three matrices share one index format. */
typedef struct vq3_mlp_layer {
  vq3_linear gate;
  vq3_linear up;
  vq3_linear down;
} vq3_mlp_layer;

/* Size in bytes of one matrix's GPU-layout indices (equal to the canonical
 * stream's size: 6 bits per output pair and input column, i.e. 3 bits per weight).
 * Cited: model card "anemll/anemll-forge-qwen3.8-27B", "Release 0.2" bullet
 * "Three bits per MLP weight" (one six-bit index per pair of output channels).
 * 0 if unsupported (d_in or d_out not a positive multiple of 64). */
VQ3_API size_t vq3_packed_bytes(int d_in, int d_out);

/*
 * Host-side, offline. Reorders a canonical index stream into the GPU layout.
 * Cited: model card "anemll/anemll-forge-qwen3.8-27B", "Release 0.2" bullet
 * "Three bits per MLP weight" (six-bit indices, one per output pair and input
 * column) and "Files and runtime compatibility" (the shipped three-bit vector
 * LUTs). The pages fix neither the index order nor the bit order; the canonical
 * stream below is the plainest reading (row-major [d_out/2][d_in] indices,
 * least significant bit first, "packed little-endian" as the workloads state).
 * canonical: host, ceil(6*(d_out/2)*d_in/8) bytes. Index k = p*d_in + i
 *   (output pair p, input column i) occupies stream bits [6k, 6k+6), stream bit
 *   j being bit (j mod 8) of byte j/8 (least significant bit first).
 * dst_host: host, vq3_packed_bytes(d_in, d_out) bytes, written in full.
 * Errors: VQ3_EINVAL (null pointer), VQ3_EUNSUPPORTED (d_in or d_out not a
 * positive multiple of 64).
 */
VQ3_API int vq3_pack_layout(const uint8_t* canonical, int d_in, int d_out, void* dst_host);

/* Host-side inverse of vq3_pack_layout (pad bits of the canonical stream are
 * written as zero), so the private GPU layout round-trips to the interchange
 * stream bit for bit. Cited: model card "anemll/anemll-forge-qwen3.8-27B",
 * "Release 0.2" bullet "Three bits per MLP weight" (one six-bit index per pair of
 * output channels and input column); the stream's order (pair-major, input
 * fastest, indices LSB-first) is this library's reading, as for vq3_pack_layout,
 * since the pages give no order. Errors as vq3_pack_layout. */
VQ3_API int vq3_unpack_layout(const void* packed_host, int d_in, int d_out, uint8_t* canonical);

/* The same three calls for any index format (VQ3_FORMAT_*): the GPU layout is
 * built from super-units of 64 output channels x 64 inputs (1536, 1024 or 2048
 * bytes), the same size as the canonical stream. An unknown format gives 0 /
 * VQ3_EUNSUPPORTED. */
VQ3_API size_t vq3_packed_bytes_fmt(int format, int d_in, int d_out);
VQ3_API int vq3_pack_layout_fmt(int format, const uint8_t* canonical, int d_in, int d_out, void* dst_host);
VQ3_API int vq3_unpack_layout_fmt(int format, const void* packed_host, int d_in, int d_out, uint8_t* canonical);

/*
 * Packed-weight blob: one matrix as a single host byte buffer (a file's contents),
 * so that a converted layer is stored once and loaded without repacking. This
 * library's own format: the pages ship their converted layers in their runtime's
 * files and do not give that layout. Host-side, offline; allocates nothing.
 * Layout (little-endian, every section at a 256-byte aligned offset):
 *   header, 256 bytes: magic "VQ3BLOB1"; version (1); d_in, d_out, block, format,
 *     lr_rank, flags (bit 0: sign bits present); offset and size of each section
 *     below; FNV-1a 64-bit hash of every byte after the header;
 *   canonical index stream (vq3_pack_layout_fmt's input, vq3_packed_bytes_fmt bytes);
 *   GPU-layout indices (vq3_pack_layout_fmt of that stream, the same size);
 *   scales FP16 [d_out]; codebook (FP16x2 [64] or [16] words, FP16 [16] for lut4);
 *   sign bits [d_in / 32] when present; U FP16 [d_out][lr_rank] and
 *   V FP16 [lr_rank][d_in] when lr_rank > 0.
 * vq3_blob_bytes: the blob's size, 0 for an unsupported descriptor.
 * vq3_blob_write: host inputs -> out (out_bytes >= vq3_blob_bytes). signs may be
 *   NULL; lr_u, lr_v are read only when lr_rank > 0. It builds the GPU layout itself.
 * vq3_blob_read: checks the magic, version, descriptor, section table, hash and
 *   that the GPU-layout section is the layout of the canonical one, then fills
 *   *view with the descriptor and host pointers into blob (valid while it is).
 * Errors: VQ3_EINVAL (null pointer, bad sizes, a blob that fails a check: the
 *   message says which), VQ3_EUNSUPPORTED (format, d_in / d_out, block, lr_rank),
 *   VQ3_ENOSPACE (out_bytes too small).
 */
typedef struct vq3_blob_view {
  int d_in, d_out, block, format, lr_rank, has_signs;
  const uint8_t* canonical;   /* vq3_packed_bytes_fmt(format, d_in, d_out) bytes */
  const void* packed;         /* the same size, GPU layout */
  const uint16_t* scales;     /* [d_out] */
  const void* codebook;       /* codebook_bytes */
  size_t codebook_bytes;
  const uint32_t* signs;      /* [d_in / 32] or NULL */
  const uint16_t* lr_u;       /* [d_out][lr_rank] or NULL */
  const uint16_t* lr_v;       /* [lr_rank][d_in] or NULL */
} vq3_blob_view;

VQ3_API size_t vq3_blob_bytes(int d_in, int d_out, int format, int lr_rank, int has_signs);
VQ3_API int vq3_blob_write(int d_in, int d_out, int block, int format, const uint8_t* canonical,
                           const uint16_t* scales, const void* codebook, const uint32_t* signs, int lr_rank,
                           const uint16_t* lr_u, const uint16_t* lr_v, void* out, size_t out_bytes);
VQ3_API int vq3_blob_read(const void* blob, size_t bytes, vq3_blob_view* view);

/*
 * Blocked, normalised fast Walsh-Hadamard transform of each row:
 *   out[r, j*b:(j+1)*b] = H_b diag(s_j) x[r, j*b:(j+1)*b] / sqrt(b).
 * Cited: model card "anemll/anemll-forge-qwen3.8-27B", "Release 0.2" bullet
 * "Token-mixer rotations" (1,024-wide Hadamard blocks with seeded signs).
 * x, out: device FP16 [rows][n]; they may alias (in place). n % block == 0,
 * block a power of two in [2, 1024]. signs: device bit-packed over n, or NULL.
 * Arithmetic in FP32, one FP16 rounding at the end.
 */
VQ3_API int fwht_rotate(const uint16_t* x, int rows, int n, int block, const uint32_t* signs,
                uint16_t* out, void* stream);

/*
 * Workspace for vq3_linear_forward / vq3_mlp_forward at `rows` rows. It holds
 * a device status word and counter words (both at fixed offsets), then
 * scratch: below 17 rows h of one pass of up to 16 rows (MLP) and the split-K
 * partial sums of both decode steps; from 17 rows on x', h, h' and the sums of
 * tiles split between CTAs. It must be zero-filled once before its first use
 * (vq3_workspace_init); every completed call leaves the counters at zero
 * again, so a workspace of the largest size needed serves calls of any row
 * count. Calls that share a workspace must not overlap on the GPU (same
 * stream, or ordered by events).
 * Device status: the first 32-bit word of the workspace stays 0. It becomes 3
 * if a wait inside a kernel gave up after its time bound (about a second); the
 * kernel still ends, the outputs of that call are invalid, and later calls on
 * the workspace skip their waits until vq3_workspace_init clears the word.
 * vq3_workspace_status copies it to the host after the stream's prior work.
 * These four calls have no counterpart on the pages: they are this library's
 * interface for caller-owned scratch.
 */
VQ3_API size_t vq3_linear_workspace_bytes(int rows, const vq3_linear* L);
VQ3_API size_t vq3_mlp_workspace_bytes(int rows, const vq3_mlp_layer* layer);
VQ3_API int vq3_workspace_init(void* workspace, size_t ws_bytes, void* stream);
VQ3_API int vq3_workspace_status(const void* workspace, int* status_host, void* stream);

/*
 * One rotated VQ3 linear layer: out = fp16( W (R x) ), FP32 accumulation.
 * Cited: model card "anemll/anemll-forge-qwen3.8-27B", "Release 0.2" bullets
 * "Three bits per MLP weight" (W = diag(scales) C[idx]) and "Token-mixer
 * rotations" (the input multiplied online by 1,024-wide Hadamard blocks with
 * seeded signs, the weights stored in the rotated basis); table row "Token
 * mixers" for the optional rank-64 factors.
 * x: device FP16 [rows][d_in]; out: device FP16 [rows][d_out] (must not alias x).
 * Errors: VQ3_EINVAL, VQ3_EALIGN, VQ3_EUNSUPPORTED, VQ3_ENOSPACE, VQ3_ECUDA.
 */
VQ3_API int vq3_linear_forward(const uint16_t* x, int rows, const vq3_linear* L, uint16_t* out,
                       void* workspace, size_t ws_bytes, void* stream);

/*
 * One SwiGLU MLP block with online rotations on both inputs:
 *   h   = silu(W_g R_g x) * (W_u R_g x)      (FP32)
 *   out = fp16( W_d R_d h )                  (R_d h rounded to FP16 once, as the MMA operand)
 * Below 17 rows: one cooperative kernel per pass of up to 8 or 16 rows;
 * all of its CTAs are resident at once and hand over between steps through
 * workspace counters. From 17 rows on: four kernels (rotate x; gate/up GEMM
 * on the tensor cores with SwiGLU fused; rotate h; down GEMM), each GEMM one
 * cooperative launch of one CTA per SM that shares out the (tile, K step)
 * pairs evenly; a tile split between CTAs is summed in K order by the CTA
 * holding its first part, so results do not depend on timing.
 * Cited: model card "anemll/anemll-forge-qwen3.8-27B", "Release 0.2" table row
 * "MLP gate / up / down" and bullets; "ANEMLL ANE LLM conversion pipeline",
 * "Facts" (SiLU form).
 * x: device FP16 [rows][d]; out: device FP16 [rows][d] (d = gate.d_in); out may
 * not alias x. Same errors as vq3_linear_forward.
 */
VQ3_API int vq3_mlp_forward(const uint16_t* x, int rows, const vq3_mlp_layer* layer, uint16_t* out,
                    void* workspace, size_t ws_bytes, void* stream);

/*
 * Gated delta-rule token mixer (the recurrent core of the pages' DeltaNet
 * layers), processed in blocks of 8 tokens with the exact closed-form block
 * inverse (I + N)^-1 = (I - N)(I + N^2)(I + N^4). Cited: model card
 * "anemll/anemll-forge-qwen3.8-27B", "Faster exact graph (previous update)",
 * bullet "Gated DeltaNet". Per head h, token t:
 *   S <- alpha[t][h] S + beta[t][h] k_t (v_t - alpha[t][h] S^T k_t)^T,   out_t = S^T q_t
 * q, k : device FP16 [tokens][heads][d_k];  v, out: device FP16 [tokens][heads][d_v]
 * beta, alpha: device FP32 [tokens][heads];  state: device FP32 [heads][d_k][d_v],
 *   read as the state before the first token and overwritten with the state after
 *   the last (FP32 accumulation, out rounded to FP16 once). With d_k a multiple of 16
 *   up to 128 and q, k, v 16-byte aligned the products run on the tensor cores, the FP32
 *   state and weighted values entering them as two FP16 parts (hi and the remainder,
 *   about 22 bits); otherwise FP32 on CUDA cores.
 * d_k a multiple of 8 in [8, 256]; d_v a multiple of 16. Deterministic.
 * Errors: VQ3_EINVAL (null pointer, bad sizes), VQ3_EUNSUPPORTED (d_k, d_v),
 * VQ3_ECUDA.
 */
VQ3_API int vq3_delta_rule_forward(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* beta,
                                   const float* alpha, int tokens, int heads, int d_k, int d_v, float* state,
                                   uint16_t* out, void* stream);

/*
 * Cited as vq3_residual_rmsnorm and vq3_mlp_forward (the two fused).
 * One layer of the pre-norm residual stack: r' = fp16(r_in + delta) (r_in alone when
 * delta is NULL), n = fp16(r' / sqrt(mean(r'^2) + eps)) per row, out = the MLP block
 * of n (as vq3_mlp_forward); r' is written to r_out. Up to 16 rows the residual
 * step runs inside the block's kernel (each CTA computes the rows' RMS; the gate/up
 * rotation normalises on the fly), from 17 rows on as a separate kernel. r_in,
 * delta: device FP16 [rows][d]; r_out, out: device FP16 [rows][d], aliasing neither
 * each other nor r_in or delta (callers alternate two residual buffers). Workspace
 * as vq3_mlp_forward. Errors as vq3_mlp_forward.
 */
VQ3_API int vq3_mlp_forward_residual(const uint16_t* r_in, const uint16_t* delta, int rows,
                                     const vq3_mlp_layer* layer, float eps, uint16_t* r_out, uint16_t* out,
                                     void* workspace, size_t ws_bytes, void* stream);

/*
 * Cited as vq3_residual_rmsnorm and vq3_mlp_forward (the two fused; the partial sums of
 * squares are this library's way to hand the next RMS over, not the pages').
 * One pre-norm MLP sublayer of the residual stack, chained through sums of squares so
 * that no kernel reads whole rows for the RMS:
 *   n      = fp16(r / sqrt(mean(r^2) + eps))   per row (unit-weight RMSNorm)
 *   out    = the MLP block of n (as vq3_mlp_forward)
 *   r_next = fp16(r + out)
 *   ss_next[row][g] = sum over columns 16g .. 16g+15 of r_next^2, each square rounded
 *                     to FP32 and added in column order
 * ss, if not NULL, holds r's partial sums in the same layout (as the previous call wrote
 * them) and the RMS is taken from them; NULL takes it from r's rows. ss_next may be NULL
 * (the partials are then not written). Up to 16 rows everything runs inside the block's
 * kernel (the residual step in its output step); from 17 rows on as an RMSNorm kernel,
 * the tensor-core path and a residual kernel. r, out, r_next: device FP16 [rows][d];
 * ss, ss_next: device FP32 [rows][d / 16]; all 16-byte aligned; out, r_next and ss_next
 * alias neither r, ss nor each other. Workspace as vq3_mlp_forward. Errors as
 * vq3_mlp_forward.
 */
VQ3_API int vq3_mlp_prenorm_step(const uint16_t* r, const float* ss, int rows, const vq3_mlp_layer* layer, float eps,
                                 uint16_t* out, uint16_t* r_next, float* ss_next, void* workspace, size_t ws_bytes,
                                 void* stream);

/* Interface query (no counterpart on the pages).
 * Number of kernels one vq3_mlp_forward call launches at `rows` rows: one per
 * pass of 8 or 16 rows below 17 rows, 4 from 17 rows on (-1 on a bad
 * descriptor). */
VQ3_API int vq3_mlp_kernel_launches(int rows, const vq3_mlp_layer* layer);

/*
 * Number of kernels one vq3_linear_forward call launches at `rows` rows: 1
 * below 17 rows (the decode kernel, which also forms the low-rank correction
 * of a layer with factors); from 17 rows on 2 (rotation, GEMM), 5 with
 * low-rank factors (plus their projection, its reduction and the expansion).
 * -1 on a bad descriptor or negative rows.
 */
VQ3_API int vq3_linear_kernel_launches(int rows, const vq3_linear* L);

/*
 * Cited as vq3_mlp_forward (an interface convenience for host buffers).
 * Same as vq3_mlp_forward with HOST buffers: copies x (pinned or pageable host
 * memory) to the workspace, runs the block, copies the result back into
 * out_host and waits for the stream. Workspace: vq3_mlp_host_workspace_bytes.
 */
VQ3_API size_t vq3_mlp_host_workspace_bytes(int rows, const vq3_mlp_layer* layer);
VQ3_API int vq3_mlp_forward_host(const uint16_t* x_host, int rows, const vq3_mlp_layer* layer,
                         uint16_t* out_host, void* workspace, size_t ws_bytes, void* stream);

/*
 * vq3_mlp_forward for callers that cannot allocate device memory. The source
 * pages have no counterpart: this is an interface convenience of this library.
 *
 * Some callers cannot call cudaMalloc at all, e.g. a plugin inside a host
 * framework that owns every device allocation, or a server that reserved its
 * whole memory budget before it started. This entry point takes no workspace:
 * its scratch is a fixed array of VQ3_NOALLOC_SCRATCH_BYTES (32 MiB) compiled
 * into the library, which every GPU that loads the library holds until the
 * process exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Size limit: any row count runs, in passes of 32, 16 or 8 rows: the
 *     largest pass whose scratch fits the array (16 rows at hidden 5120 /
 *     intermediate 17408 on a 152-SM GB300). Widths whose scratch exceeds the
 *     array even in 8-row passes return VQ3_ENOSPACE and launch nothing.
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream
 *     capture on the device.
 *   - Every call on a device shares the one array and it keeps the previous
 *     call's contents (the call clears the parts that must start at zero), so
 *     calls that overlap on the GPU race: order them on one stream or with events.
 *   - The array starts with a device status word, like a workspace. Each call
 *     clears it (with the counter words) before its kernels run; it becomes 3 if
 *     a bounded wait inside that call gave up (about a second), and that call's
 *     output is then invalid. vq3_noalloc_status reads it.
 * Arguments, output and errors otherwise as vq3_mlp_forward.
 */
#define VQ3_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
VQ3_API int vq3_mlp_forward_noalloc(const uint16_t* x, int rows, const vq3_mlp_layer* layer, uint16_t* out,
                                    void* stream);

/* Status word of the no-alloc array on the current device after the stream's prior
 * work (0, or 3 when a wait in the last vq3_mlp_forward_noalloc call gave up); copies
 * it to *status_host and waits for the stream. Allocates nothing. Errors: VQ3_EINVAL
 * (null pointer), VQ3_ECUDA. */
VQ3_API int vq3_noalloc_status(int* status_host, void* stream);

/*
 * Pre-norm residual step between stacked layers:
 *   resid  <- fp16(resid + delta)                       (skipped if delta == NULL)
 *   normed <- fp16(resid / sqrt(mean(resid^2) + eps))    (unit weight, FP32 math)
 * Cited: model card "anemll/anemll-forge-qwen3.8-27B", "Release 0.2" table row
 * "MLP gate / up / down" (the VQ3 MLP in all 64 layers of the dense model) and
 * "ANEMLL ANE LLM conversion pipeline", opening summary "Model rewrite for ANE"
 * (FP16-only graphs with a precise RMSNorm built from ANE ops). The pages give
 * neither the norm's placement nor its epsilon: pre-norm, unit weight and eps
 * inside the square root is the plainest reading, with eps = 1e-6 as the
 * stacked-layer workload states.
 * resid, delta, normed: device FP16 [rows][n]; normed may not alias resid.
 * Errors: VQ3_EINVAL (rows < 0, n <= 0, eps < 0 or NaN, null resid or normed),
 * VQ3_EALIGN (a pointer not 16-byte aligned), VQ3_ECUDA.
 */
VQ3_API int vq3_residual_rmsnorm(uint16_t* resid, const uint16_t* delta, int rows, int n, float eps,
                         uint16_t* normed, void* stream);

/*
 * Debug/test: writes the dense weight of L from its GPU layout. Cited: model card
 * "anemll/anemll-forge-qwen3.8-27B", "Release 0.2" bullet "Three bits per MLP
 * weight" (centroid component c of index idx[p][i] is the weight of output
 * channel 2p+c at input i, times that channel's scale) and "ANEMLL ANE LLM
 * conversion pipeline", "Facts" (the two-component vectors run along output
 * channels).
 * apply_scale = 0: w_out[o][i] = C[idx[o/2][i]][o%2] (exact copy of the FP16 centroid);
 * apply_scale = 1: w_out[o][i] = fp16(fp32(scale[o]) * fp32(C[...])) (the FP32
 * product is exact, so this is the correctly rounded weight).
 * w_out: device FP16 [d_out][d_in].
 */
VQ3_API int vq3_dequant_dense(const vq3_linear* L, int apply_scale, uint16_t* w_out, void* stream);

/* Message for the last error on the calling thread ("" if none). */
VQ3_API const char* vq3_last_error(void);

/* Library build/version string. */
VQ3_API const char* vq3_version(void);

/*
 * Bounds-check build (the library compiled with -DVQ3_BOUNDS_CHECK; in any other
 * build this returns VQ3_EUNSUPPORTED and writes nothing). A debugging aid of this
 * library, no counterpart on the pages. In that build every
 * global load and store of the kernels that is addressed by computed indices checks
 * the index against the extent of the buffer it addresses (the extents the entry
 * points' arguments fix); an access out of range is skipped and counted. This reads
 * the counts: out[2 f] = accesses skipped in kernel file f, out[2 f + 1] = the site
 * number of the first one (0 if none), for f = 0 decode, 1 low-rank factors,
 * 2 delta rule, 3 rotation and residual, 4 prefill up to 128 rows, 5 prefill above.
 * reset != 0 clears the counts after reading. n_out: entries of out, at least
 * VQ3_BOUNDS_FILES * 2 (else VQ3_EINVAL). Synchronous on the device (waits for all
 * work); call it between, not during, launches.
 */
#define VQ3_BOUNDS_FILES 6
VQ3_API int vq3_bounds_check(unsigned* out, int n_out, int reset);

#ifdef __cplusplus
}
#endif

#endif /* VQ3_H_ */
