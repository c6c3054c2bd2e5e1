"""Pins for the oracle's other index formats: the two-bit vector LUT ("2x16":
16 two-component centroids, a four-bit index per output pair) and the four-bit
scalar LUT ("lut4": 16 entries, a four-bit index per weight), both with
per-output-channel scales.

Source: model card "anemll/anemll-forge-qwen3.8-27B", the release-comparison
table (rows "MLP gate / up / down" and "Token mixers": two-bit vector LUT (2x16)
and four-bit LUT); "ANEMLL ANE LLM conversion pipeline", "Facts" (the previous
target mixes 2-bit vector LUTs and 4-bit scalar LUTs). Each test checks the
oracle against something other than itself: a hand-derived packing example,
weights written out by hand, a closed form, the pinned three-bit format, and the
pure-Python brute force.
"""

import math
import os

import numpy as np
import pytest

from oracle import bruteforce as bf
from oracle import vq3_oracle as O
from synth import inputs as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_pack4_golden():
    cases = []
    with open(os.path.join(GOLDEN, "canonical_pack_4bit.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, idx, byts = (p.strip() for p in line.split("|"))
            cases.append((name, [int(v) for v in idx.split()], bytes(int(b, 16) for b in byts.split())))
    return cases


@pytest.mark.parametrize("name,idx,byts", load_pack4_golden())
def test_golden_pack4_examples(name, idx, byts):
    assert O.pack_indices(np.array(idx), 4).tobytes() == byts, name
    assert O.unpack_indices(np.frombuffer(byts, np.uint8), 0, len(idx), 4).tolist() == idx
    assert [bf.index_at(byts, k, 4) for k in range(len(idx))] == idx


@pytest.mark.parametrize("n", [1, 2, 3, 7, 64, 1001])
def test_pack4_roundtrip_random(n):
    idx = np.random.default_rng(n).integers(0, 16, n)
    s = O.pack_indices(idx, 4)
    assert s.size == (4 * n + 7) // 8
    assert np.array_equal(O.unpack_indices(s, 0, n, 4), idx)
    for start in (0, n // 3, max(0, n - 2)):
        assert np.array_equal(O.unpack_indices(s, start, n - start, 4), idx[start:])


@pytest.mark.parametrize("fmt,bpw", [("2x64", 3), ("2x16", 2), ("lut4", 4)])
def test_size_arithmetic_bits_per_weight(fmt, bpw):
    d_in, d_out = 5120, 17408
    assert S.stream_bytes(d_in, d_out, fmt) * 8 == bpw * d_in * d_out


def test_dense_weight_2x16_by_hand():
    d_in, d_out = 4, 4
    idx = np.array([[1, 0, 2, 15], [15, 2, 1, 0]])  # idx[p, i]
    C = np.zeros((16, 2), np.float16)
    C[0] = (1, 10)
    C[1] = (2, 20)
    C[2] = (3, 30)
    C[15] = (4, 40)
    sc = np.array([1, 2, 0.5, 4], np.float16)
    W = O.dense_weight(O.pack_indices(idx, 4), C, sc, d_in, d_out, fmt="2x16")
    expect = np.array([[2, 1, 3, 4],
                       [40, 20, 60, 80],
                       [2, 1.5, 1, 0.5],
                       [160, 120, 80, 40]])
    assert np.array_equal(W, expect)


def test_dense_weight_lut4_by_hand():
    d_in, d_out = 3, 2
    idx = np.array([[0, 5, 15], [15, 0, 5]])  # idx[o, i]: one index per weight
    C = np.zeros((16, 1), np.float16)
    C[0, 0] = 1
    C[5, 0] = -2
    C[15, 0] = 0.25
    sc = np.array([2, 4], np.float16)
    W = O.dense_weight(O.pack_indices(idx, 4), C, sc, d_in, d_out, fmt="lut4")
    assert np.array_equal(W, np.array([[2, -4, 0.5], [1, 4, -8]]))


def test_2x16_equals_2x64_with_the_same_small_indices():
    # a two-bit vector matrix is the three-bit format restricted to the first 16
    # centroids: repacking its indices as six-bit ones gives the same weights
    d_in, d_out = 128, 64
    m = S.matrix(S.rng(30), d_in, d_out, 64, "2x16")
    idx = O.index_matrix(m.stream, d_in, d_out, fmt="2x16")
    C64 = np.zeros((64, 2), np.float16)
    C64[:16] = m.codebook
    W16 = O.dense_weight(m.stream, m.codebook, m.scales, d_in, d_out, fmt="2x16")
    W64 = O.dense_weight(O.pack_indices(idx), C64, m.scales, d_in, d_out)
    assert np.array_equal(W16, W64)


@pytest.mark.parametrize("fmt,k", [("2x16", 0), ("2x16", 11), ("lut4", 3), ("lut4", 15)])
def test_closed_form_all_indices_equal(fmt, k):
    # all indices = k, no signs: y[t, o] = s[o] C[k][o mod v] sqrt(b) sum_blocks x[t, block start]
    d_in, d_out, b = 64, 8, 16
    _, vec, _ = O.FORMATS[fmt]
    m = S.matrix(S.rng(31), d_in, d_out, b, fmt)
    m.stream = O.pack_indices(np.full((d_out // vec) * d_in, k), 4)
    x = S.activations(S.rng(32, 0), 3, d_in)
    y = O.linear_f64(x, m)
    xs = x.astype(np.float64)[:, ::b].sum(axis=1)
    C = m.codebook.astype(np.float64)
    sc = m.scales.astype(np.float64)
    expect = np.stack([sc[o] * C[k][o % vec] * math.sqrt(b) * xs for o in range(d_out)], axis=1)
    assert np.allclose(y, expect, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("fmt", ["2x16", "lut4"])
@pytest.mark.parametrize("d_in,d_out,T,block,signs", [(2, 2, 1, 2, False), (8, 4, 3, 4, True), (4, 4, 2, 2, False)])
def test_bruteforce_linear(fmt, d_in, d_out, T, block, signs):
    m = S.matrix(S.rng(40 + d_in), d_in, d_out, block, fmt)
    if signs:
        m.signs = S.sign_bits(S.rng(40 + d_in, 2), d_in)
    x = S.activations(S.rng(41, 0), T, d_in)
    assert np.allclose(O.linear_f64(x, m), np.array(bf.linear(x.tolist(), m)), rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("fmt", ["2x16", "lut4"])
def test_bruteforce_mlp(fmt):
    blk = S.mlp_block(S.rng(50), 4, 8, 4, fmt)
    S.add_signs(S.rng(50, 2), blk)
    x = S.activations(S.rng(51, 0), 2, 4)
    assert np.allclose(O.mlp_f64(x, blk), np.array(bf.mlp(x.tolist(), blk)), rtol=1e-10, atol=1e-15)


def test_planted_mistakes_are_caught():
    # reading a four-bit stream with the six-bit width breaks the golden example
    _, idx, byts = load_pack4_golden()[0]
    assert O.unpack_indices(np.frombuffer(byts, np.uint8), 0, 2, 6).tolist() != idx[:2]
    # reading a scalar matrix as a vector one (two channels per index) breaks the hand layout
    idx = np.array([[0, 5, 15], [15, 0, 5]])
    C = np.zeros((16, 2), np.float16)
    C[:, 0] = np.arange(16)
    C[:, 1] = -np.arange(16)
    W_vec = O.dense_weight(O.pack_indices(idx, 4), C, np.ones(2, np.float16), 3, 2, fmt="2x16")
    W_sc = O.dense_weight(O.pack_indices(idx, 4), C[:, :1], np.ones(2, np.float16), 3, 2, fmt="lut4")
    assert not np.array_equal(W_vec, W_sc)
