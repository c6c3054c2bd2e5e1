"""Seeded synthetic inputs for the VQ3 Hadamard-rotated vector-LUT MLP.

This module is shared by the CPU oracle tests and by the CUDA path's tests and
benchmark. It draws random numbers and nothing else: it holds none of the
method's arithmetic (no unpacking, no rotation, no lookup, no matmul).

The index stream is drawn directly in its canonical form. Uniform random 6-bit
indices packed back to back are uniformly random bits, so the stream is random
bytes whose pad bits (past the last index) are cleared. Both sides unpack it
with their own code.

Each workload seed feeds three independent PCG64 streams (seed sequences
[seed, 0], [seed, 1] and [seed, 2]): activations, weights and sign bits. The
weights therefore do not depend on the row count, so a row sweep runs the same
block at every T, and the first rows of a taller X equal a shorter X. Inside the
weight stream the order is fixed: for each matrix in order (gate, up, down for a
block; layer by layer for a stack) the codebook, then the index stream, then the
scales.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HIDDEN = 5120
INTERMEDIATE = 17408
CODEBOOK_SIZE = 64
CENTROID_DIM = 2
INDEX_BITS = 6

# index format -> (index bits, centroid dimension, codebook entries); "2x64" is the
# three-bit vector format, "2x16" the two-bit vector format, "lut4" the four-bit
# scalar format
FORMATS = {"2x64": (6, 2, 64), "2x16": (4, 2, 16), "lut4": (4, 1, 16)}


def rng(seed: int, stream: int = 1) -> np.random.Generator:
    """Stream 0: activations; 1: weights; 2: sign bits."""
    return np.random.Generator(np.random.PCG64([seed, stream]))


def stream_bytes(d_in: int, d_out: int, fmt: str = "2x64") -> int:
    """Length in bytes of the canonical stream of a d_out x d_in matrix."""
    nb, vec, _ = FORMATS[fmt]
    bits = nb * (d_out // vec) * d_in
    return (bits + 7) // 8


def activations(g: np.random.Generator, rows: int, n: int, outlier_channels: int = 0,
                outlier_scale: float = 50.0) -> np.ndarray:
    """FP16 activations ~N(0,1); optionally `outlier_channels` seeded columns scaled up."""
    x = g.standard_normal((rows, n), dtype=np.float64)
    if outlier_channels:
        cols = np.sort(g.choice(n, size=outlier_channels, replace=False))
        x[:, cols] *= outlier_scale
    return x.astype(np.float16)


def codebook(g: np.random.Generator, std: float = 0.02, fmt: str = "2x64") -> np.ndarray:
    """FP16 codebook [entries, centroid dim] ~N(0, std) ([64, 2] for "2x64")."""
    _, vec, entries = FORMATS[fmt]
    return (g.standard_normal((entries, vec)) * std).astype(np.float16)


def index_stream(g: np.random.Generator, d_in: int, d_out: int, fmt: str = "2x64") -> np.ndarray:
    """Canonical index stream of uniformly random indices (uint8 bytes)."""
    nb, vec, _ = FORMATS[fmt]
    nbytes = stream_bytes(d_in, d_out, fmt)
    s = g.integers(0, 256, size=nbytes, dtype=np.uint8)
    tail_bits = (nb * (d_out // vec) * d_in) % 8
    if tail_bits:
        s[-1] &= np.uint8((1 << tail_bits) - 1)
    return s


def scales(g: np.random.Generator, d_out: int, lo: float = 0.5, hi: float = 1.5) -> np.ndarray:
    """FP16 per-output-channel scales ~U[lo, hi]."""
    return g.uniform(lo, hi, size=d_out).astype(np.float16)


def sign_bits(g: np.random.Generator, n: int) -> np.ndarray:
    """Bit-packed seeded signs: bit j of word j//32 set means channel j is negated."""
    words = (n + 31) // 32
    w = g.integers(0, 2**32, size=words, dtype=np.uint64).astype(np.uint32)
    tail = n % 32
    if tail:
        w[-1] &= np.uint32((1 << tail) - 1)
    return w


@dataclass
class Matrix:
    """One VQ3 matrix, d_out x d_in, in its canonical (interchange) form."""
    d_in: int
    d_out: int
    block: int
    codebook: np.ndarray  # [entries, centroid dim] float16 ([64, 2] for "2x64")
    stream: np.ndarray    # canonical LE index stream, uint8
    scales: np.ndarray    # [d_out] float16
    signs: np.ndarray | None = None  # bit-packed uint32 over d_in, or None (all +1)
    fmt: str = "2x64"     # index format (FORMATS)
    lr_u: np.ndarray | None = None  # low-rank factor U [d_out, r] float16, or None
    lr_v: np.ndarray | None = None  # low-rank factor V [r, d_in] float16


@dataclass
class Block:
    gate: Matrix
    up: Matrix
    down: Matrix


@dataclass
class Workload:
    name: str
    seed: int
    x: np.ndarray  # [rows, d] float16
    layers: list = field(default_factory=list)  # list[Block] or [Matrix]


def matrix(g: np.random.Generator, d_in: int, d_out: int, block: int, fmt: str = "2x64") -> Matrix:
    c = codebook(g, fmt=fmt)
    s = index_stream(g, d_in, d_out, fmt)
    sc = scales(g, d_out)
    return Matrix(d_in, d_out, block, c, s, sc, None, fmt)


def mlp_block(g: np.random.Generator, hidden: int, inter: int, block: int, fmt: str = "2x64") -> Block:
    gate = matrix(g, hidden, inter, block, fmt)
    up = matrix(g, hidden, inter, block, fmt)
    down = matrix(g, inter, hidden, block, fmt)
    return Block(gate, up, down)


def add_lowrank(g: np.random.Generator, m: Matrix, rank: int = 64, std: float = 0.01) -> Matrix:
    """Seeded FP16 low-rank factors U [d_out, rank], V [rank, d_in] ~N(0, std) (drawn U then V;
    callers pass a stream of its own, [seed, 3], so the other inputs do not move)."""
    m.lr_u = (g.standard_normal((m.d_out, rank)) * std).astype(np.float16)
    m.lr_v = (g.standard_normal((rank, m.d_in)) * std).astype(np.float16)
    return m


def add_signs(g: np.random.Generator, blk: Block) -> Block:
    """Seeded sign vectors: one shared by gate and up (same input), one for down."""
    s_in = sign_bits(g, blk.gate.d_in)
    s_dn = sign_bits(g, blk.down.d_in)
    blk.gate.signs = s_in
    blk.up.signs = s_in
    blk.down.signs = s_dn
    return blk


# ---- the five workloads (sizes and distributions as the benchmark specifies) ----

def linear_256(seed: int = 0, rows: int = 8) -> Workload:
    """A single VQ3 linear, 256 -> 256, one 256-point rotation block, 8 rows."""
    x = activations(rng(seed, 0), rows, 256)
    m = matrix(rng(seed, 1), 256, 256, 256)
    return Workload("linear_256x256_T8", seed, x, [m])


def mlp_27b(seed: int = 1, rows: int = 8, outlier_channels: int = 0, hidden: int = HIDDEN,
            inter: int = INTERMEDIATE, block: int = 1024, name: str | None = None, fmt: str = "2x64") -> Workload:
    """One SwiGLU block at the 27B-dense shape (hidden 5120, intermediate 17408)."""
    x = activations(rng(seed, 0), rows, hidden, outlier_channels=outlier_channels)
    blk = mlp_block(rng(seed, 1), hidden, inter, block, fmt)
    suffix = "" if fmt == "2x64" else f"_{fmt}"
    return Workload(name or f"mlp_{hidden}x{inter}_T{rows}{suffix}", seed, x, [blk])


def mlp_prefill_outliers(seed: int = 2, rows: int = 64) -> Workload:
    """Config of 64 prefill rows with 1% of the 5120 channels (51) scaled x50."""
    return mlp_27b(seed=seed, rows=rows, outlier_channels=round(0.01 * HIDDEN),
                   name=f"mlp_5120x17408_T{rows}_outliers")


def mlp_stack(seed: int = 3, rows: int = 8, layers: int = 64, hidden: int = HIDDEN,
              inter: int = INTERMEDIATE, block: int = 1024) -> Workload:
    """`layers` independent MLP blocks with a residual stream of `rows` rows."""
    x = activations(rng(seed, 0), rows, hidden)
    g = rng(seed, 1)
    blocks = [mlp_block(g, hidden, inter, block) for _ in range(layers)]
    return Workload(f"mlp_stack{layers}_{hidden}x{inter}_T{rows}", seed, x, blocks)


def mlp_sweep(seed: int = 4, rows: int = 8) -> Workload:
    """Row-sweep workload: the same block shape at T in {1, 8, 64, 512, 2048, 4096}."""
    return mlp_27b(seed=seed, rows=rows, name=f"mlp_5120x17408_T{rows}_sweep")


SWEEP_ROWS = (1, 8, 64, 512, 2048, 4096)


# the previous release's MLP formats at the same shape: seed 5 for "2x16", 6 for "lut4"
FORMAT_SEEDS = {"2x16": 5, "lut4": 6}


def mlp_format(fmt: str, rows: int = 8) -> Workload:
    """One block at 5120/17408 in another index format (two-bit vector or four-bit scalar LUT)."""
    return mlp_27b(seed=FORMAT_SEEDS[fmt], rows=rows, fmt=fmt)


# ---- gated delta-rule token mixer (the 8-row block of the pages' DeltaNet layers) ----

@dataclass
class DeltaRuleInputs:
    q: np.ndarray      # [T, H, d_k] float16
    k: np.ndarray      # [T, H, d_k] float16, rows of unit length (up to FP16 rounding)
    v: np.ndarray      # [T, H, d_v] float16
    beta: np.ndarray   # [T, H] float32 in (0, 1): write strength
    alpha: np.ndarray  # [T, H] float32 in (0, 1]: decay gate
    state: np.ndarray  # [H, d_k, d_v] float32: state before the first token


def delta_rule_inputs(seed: int = 9, tokens: int = 8, heads: int = 16, d_k: int = 128, d_v: int = 128) -> DeltaRuleInputs:
    """Seeded inputs of the delta-rule block: queries, keys (unit rows, as the layer
    normalises them) and values ~N(0,1) from stream [seed, 0]; strengths ~U[0.05, 0.95] and
    gates ~U[0.9, 1] from [seed, 1]; the initial state ~N(0, 0.1) from [seed, 2]. Head counts
    and widths are not on the pages: the defaults are synthetic."""
    g = rng(seed, 0)
    q = g.standard_normal((tokens, heads, d_k))
    k = g.standard_normal((tokens, heads, d_k))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = g.standard_normal((tokens, heads, d_v))
    gg = rng(seed, 1)
    beta = gg.uniform(0.05, 0.95, (tokens, heads)).astype(np.float32)
    alpha = gg.uniform(0.9, 1.0, (tokens, heads)).astype(np.float32)
    state = (rng(seed, 2).standard_normal((heads, d_k, d_v)) * 0.1).astype(np.float32)
    return DeltaRuleInputs(q.astype(np.float16), k.astype(np.float16), v.astype(np.float16), beta, alpha, state)
