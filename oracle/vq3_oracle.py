"""CPU oracle for the VQ3 Hadamard-rotated vector-LUT SwiGLU MLP.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports or calls this
module; only the tests, `__graft_entry__.smoke()` and the benchmark's CPU
baseline leg do. It shares no code with the CUDA library: it unpacks the
canonical stream, builds dense weights, and applies the rotation as an explicit
normalised +-1 matrix, all in NumPy float64, in the order the method defines.

Sources (page title, then section):
  [R02]   model card "anemll/anemll-forge-qwen3.8-27B", section
          "Release 0.2: three-bit MLP, token-mixer rotations, distilled weights"
          (table row "MLP gate / up / down": three-bit vector LUT (2x64); bullet
          "Three bits per MLP weight": 64 two-component centroids per matrix,
          one six-bit index per pair of output channels, per-channel scales;
          bullet "Token-mixer rotations": 1,024-wide Hadamard blocks with seeded
          signs, weights stored in the rotated basis, as the MLP already did).
  [FILES] same card, section "Files and runtime compatibility" (per-channel
          scaling and online Hadamard rotations on the MLP inputs).
  [FACTS] "ANEMLL ANE LLM conversion pipeline", section "Facts" (SiLU written
          as 0.5*x*(1+tanh(x/2)); vector LUTs along input channels lost
          placement, so the vectors run along output channels).
  [R01]   same model card, the release-comparison table (row "MLP gate / up /
          down": two-bit vector LUT (2x16) in 38 layers, four-bit LUT in 26, in
          the previous release; row "Token mixers": two-bit vector LUT and
          four-bit LUT) and "ANEMLL ANE LLM conversion pipeline", "Facts" (the
          previous target mixes 2-bit vector LUTs and 4-bit scalar LUTs).

Low-rank correction ([R01] row "Token mixers": rank-64 factors; "ANEMLL ANE
LLM conversion pipeline", "Facts": rank-64 residual correction): a matrix may
carry FP16 factors U [d_out, r] and V [r, d_in]; its weight is then
diag(s) C[idx] + U V, the factors acting on the same rotated input as the
lookup-table part and the scales on the lookup-table part only.

Index formats (FORMATS): "2x64" is the release's three-bit format (64
two-component centroids, a six-bit index per output pair); "2x16" the two-bit
vector format (16 two-component centroids, a four-bit index per output pair);
"lut4" the four-bit scalar format (16 scalar entries, a four-bit index per
weight). Every format has per-output-channel scales.

Readings where the pages are silent (each also listed in the design notes):
  * index k = p*d_in + i (group-major, input fastest; a group is an output pair
    for the vector formats, one output channel for "lut4") occupies stream bits
    [b k, b k + b) for index width b; stream bit j is bit (j mod 8) of byte j//8
    (LSB first);
  * centroid component c of index idx[p, i] is the weight of output channel
    2p+c at input column i (the single entry, of channel p, for "lut4"); the
    scale multiplies after the lookup;
  * the rotation of a row is x' = blockdiag(H_b diag(s)) x / sqrt(b), with H_b
    the Sylvester Hadamard matrix H[r][c] = (-1)^popcount(r & c) and s = +1
    unless seed signs are given; gate and up share x', down has its own;
  * SiLU(z) = z / (1 + exp(-z)), identical to the pages' tanh form.

Parity pins: every function here is pinned by tests in tests/test_oracle_pins.py
and, for the "2x16" and "lut4" formats, tests/test_oracle_formats.py (closed
forms, invariants, hand-derived packing examples, weights written out by hand
and a pure-Python brute force in oracle/bruteforce.py). No function is "parity unpinned" except
the whole-model quality figures, which need trained weights and are not
computed here.
"""

from __future__ import annotations

import functools
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

INDEX_BITS = 6
CODEBOOK_SIZE = 64

# format -> (index bits, centroid dimension = output channels per index, codebook entries)
FORMATS = {"2x64": (6, 2, 64), "2x16": (4, 2, 16), "lut4": (4, 1, 16)}


def fmt_of(m) -> str:
    """Format of a matrix object (the release's 2x64 when it names none)."""
    return getattr(m, "fmt", "2x64") or "2x64"


# ---------------------------------------------------------------------------
# canonical index stream  ([R02] "Three bits per MLP weight")
# ---------------------------------------------------------------------------

def unpack_indices(stream: np.ndarray, start: int, count: int, bits_per: int = INDEX_BITS) -> np.ndarray:
    """Indices start .. start+count-1 of a canonical stream, as int64.

    Index k occupies bits [b k, b k + b) of the stream (b = bits_per), least
    significant bit first.
    """
    stream = np.asarray(stream, dtype=np.uint8)
    first_bit = bits_per * start
    last_bit = bits_per * (start + count)
    b0 = first_bit // 8
    b1 = (last_bit + 7) // 8
    bits = np.unpackbits(stream[b0:b1], bitorder="little")
    skip = first_bit - 8 * b0
    bits = bits[skip: skip + bits_per * count].reshape(count, bits_per)
    idx = np.zeros(count, dtype=np.int64)
    for b in range(bits_per):
        idx |= bits[:, b].astype(np.int64) << b
    return idx


def pack_indices(idx: np.ndarray, bits_per: int = INDEX_BITS) -> np.ndarray:
    """Inverse of unpack_indices for a whole stream (pad bits zero)."""
    idx = np.asarray(idx, dtype=np.int64).reshape(-1)
    if idx.size and (idx.min() < 0 or idx.max() >= (1 << bits_per)):
        raise ValueError(f"indices must lie in [0, {1 << bits_per})")
    bits = ((idx[:, None] >> np.arange(bits_per)) & 1).astype(np.uint8).reshape(-1)
    pad = (-bits.size) % 8
    if pad:
        bits = np.concatenate([bits, np.zeros(pad, np.uint8)])
    return np.packbits(bits, bitorder="little")


def index_matrix(stream: np.ndarray, d_in: int, d_out: int, p0: int = 0, p1: int | None = None,
                 fmt: str = "2x64") -> np.ndarray:
    """idx[p, i] for output groups p0 <= p < p1 (default: all d_out / vec groups)."""
    bits_per, vec, _ = FORMATS[fmt]
    if p1 is None:
        p1 = d_out // vec
    return unpack_indices(stream, p0 * d_in, (p1 - p0) * d_in, bits_per).reshape(p1 - p0, d_in)


# ---------------------------------------------------------------------------
# dense weights  ([R02] codebook of 2-vectors along output-channel pairs, [FACTS])
# ---------------------------------------------------------------------------

def dense_weight(stream, codebook, scales, d_in: int, d_out: int, apply_scale: bool = True,
                 rows: tuple[int, int] | None = None, fmt: str = "2x64") -> np.ndarray:
    """W[v p + c, i] = scale[v p + c] * C[idx[p, i]][c] in float64 (v = centroid
    dimension: 2 for the vector formats, 1 for "lut4"), for output rows [r0, r1).

    Both factors are FP16; their product is exact in float64 (and in float32).
    """
    _, vec, entries = FORMATS[fmt]
    r0, r1 = (0, d_out) if rows is None else rows
    if r0 % vec or r1 % vec:
        raise ValueError("row range must cover whole output-channel groups")
    idx = index_matrix(stream, d_in, d_out, r0 // vec, r1 // vec, fmt)
    C = np.asarray(codebook, dtype=np.float16).astype(np.float64).reshape(entries, vec)
    W = np.empty((r1 - r0, d_in), dtype=np.float64)
    for c in range(vec):
        W[c::vec, :] = C[idx, c]
    if apply_scale:
        W *= np.asarray(scales, dtype=np.float16).astype(np.float64)[r0:r1, None]
    return W


# ---------------------------------------------------------------------------
# rotation  ([R02] "Token-mixer rotations", [FILES])
# ---------------------------------------------------------------------------

def popcount_parity(m: np.ndarray) -> np.ndarray:
    m = np.asarray(m, dtype=np.int64)
    parity = np.zeros_like(m)
    while np.any(m):
        parity ^= m & 1
        m = m >> 1
    return parity


@functools.lru_cache(maxsize=16)
def hadamard(b: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order b (a power of two): H[r][c] = (-1)^popcount(r & c).

    The returned array is cached and read-only."""
    if b < 1 or b & (b - 1):
        raise ValueError("Hadamard order must be a power of two")
    r = np.arange(b)
    H = 1.0 - 2.0 * popcount_parity(r[:, None] & r[None, :]).astype(np.float64)
    H.setflags(write=False)
    return H


def sign_vector(sign_words, n: int) -> np.ndarray:
    """+-1 vector from bit-packed sign words (bit set = -1); None means all +1."""
    if sign_words is None:
        return np.ones(n, dtype=np.float64)
    w = np.asarray(sign_words, dtype=np.uint32)
    j = np.arange(n)
    bit = (w[j // 32] >> (j % 32).astype(np.uint32)) & 1
    return 1.0 - 2.0 * bit.astype(np.float64)


def rotation_block(b: int, s: np.ndarray | None = None) -> np.ndarray:
    """One diagonal block of the rotation: H_b diag(s) / sqrt(b)."""
    H = hadamard(b)
    if s is not None:
        H = H * np.asarray(s, dtype=np.float64)[None, :]
    return H / math.sqrt(b)


def rotate(x: np.ndarray, block: int, sign_words=None) -> np.ndarray:
    """x' = blockdiag(H_b diag(s)) x / sqrt(b) for every row of x, in float64."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    if n % block:
        raise ValueError("row length must be a multiple of the rotation block")
    s = sign_vector(sign_words, n)
    out = np.empty_like(x)
    for j in range(n // block):
        sl = slice(j * block, (j + 1) * block)
        R = rotation_block(block, s[sl])
        out[..., sl] = x[..., sl] @ R.T
    return out


# ---------------------------------------------------------------------------
# forward passes
# ---------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + exp(-z)); equal to 0.5 z (1 + tanh(z/2)) ([FACTS])."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def _as_f16_f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float16).astype(np.float64)


def lowrank_f64(xr, m) -> np.ndarray | None:
    """U (V x') for the rotated rows xr of a matrix with low-rank factors, else None."""
    U = getattr(m, "lr_u", None)
    V = getattr(m, "lr_v", None)
    if U is None or V is None:
        return None
    z = np.asarray(xr, np.float64) @ _as_f16_f64(V).T
    return z @ _as_f16_f64(U).T


def linear_f64(x, m, row_chunk: int = 2048, workers: int = 1) -> np.ndarray:
    """y = W (R x) in float64 for one VQ3 matrix `m` (fields as in synth.inputs.Matrix),
    plus U (V R x) when the matrix carries low-rank factors.

    x is taken at its own precision (FP16 inputs convert exactly); nothing is rounded.
    The output channels are computed in ranges of `row_chunk`; with workers > 1 the
    ranges run on that many threads (each output is computed the same way either way).
    """
    xr = rotate(np.asarray(x, dtype=np.float64), m.block, m.signs)
    y = np.empty((xr.shape[0], m.d_out), dtype=np.float64)

    def out_range(r0):
        r1 = min(m.d_out, r0 + row_chunk)
        W = dense_weight(m.stream, m.codebook, m.scales, m.d_in, m.d_out, rows=(r0, r1), fmt=fmt_of(m))
        y[:, r0:r1] = xr @ W.T

    starts = range(0, m.d_out, row_chunk)
    if workers > 1:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(out_range, starts))
    else:
        for r0 in starts:
            out_range(r0)
    lr = lowrank_f64(xr, m)
    if lr is not None:
        y += lr
    return y


def linear(x, m) -> np.ndarray:
    """FP16 output of one rotated VQ3 linear layer (round to nearest even once)."""
    return linear_f64(x, m).astype(np.float16)


def mlp_f64(x, blk, workers: int = 1) -> np.ndarray:
    """SwiGLU block: y = W_d R_d (silu(W_g R x) * (W_u R x)), float64 throughout."""
    g = linear_f64(x, blk.gate, workers=workers)
    u = linear_f64(x, blk.up, workers=workers)
    h = silu(g) * u
    return linear_f64(h, blk.down, workers=workers)


def mlp(x, blk, workers: int = 1) -> np.ndarray:
    return mlp_f64(x, blk, workers).astype(np.float16)


def rmsnorm(r, eps: float = 1e-6) -> np.ndarray:
    """Unit-weight RMSNorm of each row, float64 math, FP16 result."""
    r = _as_f16_f64(r)
    return (r / np.sqrt(np.mean(r * r, axis=-1, keepdims=True) + eps)).astype(np.float16)


def residual_add(r, delta) -> np.ndarray:
    return (_as_f16_f64(r) + _as_f16_f64(delta)).astype(np.float16)


def stack(x, blocks, eps: float = 1e-6, trace: list | None = None, workers: int = 1) -> np.ndarray:
    """Pre-norm residual stack: r <- fp16(r + fp16(MLP_l(fp16(RMSNorm(r))))) for each layer.

    `blocks` may be any iterable (a generator keeps one layer in host memory at a time)."""
    r = np.asarray(x, dtype=np.float16)
    if trace is not None:
        trace.append(r.copy())
    for blk in blocks:
        n = rmsnorm(r, eps)
        r = residual_add(r, mlp(n, blk, workers))
        if trace is not None:
            trace.append(r.copy())
    return r


# ---------------------------------------------------------------------------
# comparison metrics used by the parity gates
# ---------------------------------------------------------------------------

def rel_max_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / denom) if denom > 0 else float(np.max(np.abs(got)))


def row_cosine(got, ref) -> np.ndarray:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.sum(got * ref, axis=-1)
    den = np.sqrt(np.sum(got * got, axis=-1) * np.sum(ref * ref, axis=-1))
    out = np.ones_like(num)
    nz = den > 0
    out[nz] = num[nz] / den[nz]
    both_zero = (den == 0) & (np.sum(got * got, axis=-1) == 0) & (np.sum(ref * ref, axis=-1) == 0)
    out[~nz & ~both_zero] = 0.0
    return out
