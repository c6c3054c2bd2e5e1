"""Pure-Python scalar brute force for tiny VQ3 shapes (test infrastructure only).

Written independently of oracle/vq3_oracle.py: no NumPy, every quantity from its
scalar definition (bit reads of the stream, Hadamard entries from the parity of
popcount(r & c), SiLU through math.exp, sums in Python floats). It serves as a
pin for the NumPy oracle on shapes small enough for scalar loops.

Index formats as in the oracle module ("2x64", "2x16", "lut4"). Sources as in the oracle module: model card "anemll/anemll-forge-qwen3.8-27B",
section "Release 0.2: three-bit MLP, token-mixer rotations, distilled weights";
"ANEMLL ANE LLM conversion pipeline", section "Facts".
"""

from __future__ import annotations

import math


def stream_bit(stream, j: int) -> int:
    return (int(stream[j // 8]) >> (j % 8)) & 1


# format -> (index bits, output channels per index)
_FMT = {"2x64": (6, 2), "2x16": (4, 2), "lut4": (4, 1)}


def index_at(stream, k: int, bits: int = 6) -> int:
    v = 0
    for b in range(bits):
        v |= stream_bit(stream, bits * k + b) << b
    return v


def had(r: int, c: int) -> int:
    return -1 if bin(r & c).count("1") % 2 else 1


def sign_at(sign_words, j: int) -> int:
    if sign_words is None:
        return 1
    return -1 if (int(sign_words[j // 32]) >> (j % 32)) & 1 else 1


def rotate_row(x, block: int, sign_words=None):
    n = len(x)
    out = [0.0] * n
    inv = 1.0 / math.sqrt(block)
    for j0 in range(0, n, block):
        for r in range(block):
            acc = 0.0
            for c in range(block):
                acc += had(r, c) * sign_at(sign_words, j0 + c) * float(x[j0 + c])
            out[j0 + r] = acc * inv
    return out


def weight(m, o: int, i: int) -> float:
    bits, vec = _FMT[getattr(m, "fmt", "2x64") or "2x64"]
    p, c = divmod(o, vec)
    k = index_at(m.stream, p * m.d_in + i, bits)
    entry = m.codebook[k]
    w = float(m.scales[o]) * float(entry[c] if vec > 1 else (entry[0] if hasattr(entry, "__len__") else entry))
    U = getattr(m, "lr_u", None)
    V = getattr(m, "lr_v", None)
    if U is not None and V is not None:
        # low-rank correction: + sum_j U[o][j] V[j][i]
        for j in range(len(V)):
            w += float(U[o][j]) * float(V[j][i])
    return w


def linear_row(x, m):
    xr = rotate_row(x, m.block, m.signs)
    return [sum(weight(m, o, i) * xr[i] for i in range(m.d_in)) for o in range(m.d_out)]


def silu(z: float) -> float:
    return z / (1.0 + math.exp(-z))


def mlp_row(x, blk):
    g = linear_row(x, blk.gate)
    u = linear_row(x, blk.up)
    h = [silu(a) * b for a, b in zip(g, u)]
    return linear_row(h, blk.down)


def linear(xs, m):
    return [linear_row(list(row), m) for row in xs]


def mlp(xs, blk):
    return [mlp_row(list(row), blk) for row in xs]
