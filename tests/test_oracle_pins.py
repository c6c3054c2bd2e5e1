"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a hand-derived
packing example, closed forms of the Hadamard transform, invariants of the
codebook format, special cases with a known answer, and a pure-Python scalar
brute force on tiny shapes. A planted-mistake section at the end shows that
plausible errors in the oracle fail at least one pin.
"""

import math
import os

import numpy as np
import pytest

from oracle import bruteforce as bf
from oracle import vq3_oracle as O
from synth import inputs as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_pack_golden():
    cases = []
    with open(os.path.join(GOLDEN, "canonical_pack.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, idx, byts = (p.strip() for p in line.split("|"))
            cases.append((name, [int(v) for v in idx.split()], bytes(int(b, 16) for b in byts.split())))
    return cases


# ---------------------------------------------------------------- packing

@pytest.mark.parametrize("name,idx,byts", load_pack_golden())
def test_golden_pack_examples(name, idx, byts):
    got = O.pack_indices(np.array(idx)).tobytes()
    assert got == byts, name
    back = O.unpack_indices(np.frombuffer(byts, np.uint8), 0, len(idx))
    assert back.tolist() == idx
    # the scalar reader agrees bit by bit
    assert [bf.index_at(byts, k) for k in range(len(idx))] == idx


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 64, 1001, 4096])
def test_pack_unpack_roundtrip_random(n):
    g = np.random.default_rng(n)
    idx = g.integers(0, 64, n)
    s = O.pack_indices(idx)
    assert s.size == (6 * n + 7) // 8
    assert np.array_equal(O.unpack_indices(s, 0, n), idx)
    # any window decodes to the same values
    for start in (0, n // 3, max(0, n - 2)):
        cnt = n - start
        assert np.array_equal(O.unpack_indices(s, start, cnt), idx[start:])


@pytest.mark.parametrize("pattern", ["zeros", "ones63", "alternate", "ramp"])
def test_pack_edge_patterns(pattern):
    n = 37
    idx = {"zeros": np.zeros(n, int), "ones63": np.full(n, 63), "alternate": np.arange(n) % 2 * 63,
           "ramp": np.arange(n) % 64}[pattern]
    s = O.pack_indices(idx)
    if pattern == "zeros":
        assert not s.any()
    if pattern == "ones63":
        # every index bit set, pad bits clear
        assert s[:-1].tolist() == [255] * (s.size - 1)
        assert s[-1] == (1 << ((6 * n) % 8 or 8)) - 1
    assert np.array_equal(O.unpack_indices(s, 0, n), idx)


def test_generator_stream_is_uniform_indices():
    g = S.rng(123)
    s = S.index_stream(g, 256, 64)
    assert s.size == S.stream_bytes(256, 64) == 6 * 32 * 256 // 8
    idx = O.unpack_indices(s, 0, 32 * 256)
    counts = np.bincount(idx, minlength=64)
    assert counts.min() > 0.6 * counts.mean() and counts.max() < 1.4 * counts.mean()


def test_size_arithmetic_three_bits_per_weight():
    # "Three bits per MLP weight": 6 bits per output pair and input column
    assert S.stream_bytes(5120, 17408) == 33_423_360
    assert S.stream_bytes(17408, 5120) == 33_423_360
    block = 3 * 33_423_360 + 2 * (17408 + 17408 + 5120) + 3 * 64 * 2 * 2
    assert block == 100_350_720
    assert 64 * block == 6_422_446_080
    assert S.stream_bytes(5120, 17408) * 8 / (5120 * 17408) == 3.0


# ---------------------------------------------------------------- Hadamard

@pytest.mark.parametrize("b", [1, 2, 4, 8, 16, 64, 256, 1024])
def test_hadamard_orthogonal(b):
    H = O.hadamard(b)
    assert np.array_equal(H @ H.T, b * np.eye(b))
    assert set(np.unique(H).tolist()) <= {-1.0, 1.0}
    assert np.array_equal(H, H.T)


def test_hadamard_sylvester_recursion():
    # H_2n = [[H_n, H_n], [H_n, -H_n]] (textbook Sylvester construction)
    for n in (1, 2, 4, 32, 512):
        H = O.hadamard(n)
        H2 = np.block([[H, H], [H, -H]])
        assert np.array_equal(O.hadamard(2 * n), H2)


@pytest.mark.parametrize("b", [4, 256, 1024])
def test_double_rotation_identity(b):
    g = np.random.default_rng(b)
    x = g.standard_normal((3, 2 * b))
    assert np.allclose(O.rotate(O.rotate(x, b), b), x, atol=1e-12)


@pytest.mark.parametrize("b", [8, 1024])
def test_signed_rotation_orthogonal_and_inverse(b):
    g = np.random.default_rng(7)
    s_words = S.sign_bits(g, b)
    s = O.sign_vector(s_words, b)
    R = O.rotation_block(b, s)
    assert np.allclose(R @ R.T, np.eye(b), atol=1e-12)
    Rinv = np.diag(s) @ O.hadamard(b) / math.sqrt(b)
    assert np.allclose(Rinv @ R, np.eye(b), atol=1e-12)
    x = g.standard_normal((2, b))
    assert np.allclose(O.rotate(x, b, s_words) @ Rinv.T, x, atol=1e-12)


def test_sign_bits_meaning():
    # bit j of word j/32 set => input j negated
    w = np.array([0b101, 1 << 31], dtype=np.uint32)
    s = O.sign_vector(w, 64)
    assert s[0] == -1 and s[1] == 1 and s[2] == -1 and s[63] == -1 and s[32] == 1


@pytest.mark.parametrize("b", [16, 1024])
def test_fwht_unit_vectors_and_constant(b):
    for j in (0, 1, b // 2 + 3, b - 1):
        e = np.zeros((1, b))
        e[0, j] = 1.0
        # transform of e_j is column j of H, divided by sqrt(b)
        assert np.allclose(O.rotate(e, b)[0], O.hadamard(b)[:, j] / math.sqrt(b), atol=0)
    c = 0.75
    out = O.rotate(np.full((1, b), c), b)[0]
    expect = np.zeros(b)
    expect[0] = c * math.sqrt(b)
    assert np.allclose(out, expect, atol=1e-12)


def test_rotation_acts_per_block():
    b = 8
    x = np.zeros((1, 3 * b))
    x[0, b:2 * b] = np.arange(1, b + 1)
    out = O.rotate(x, b)
    assert not out[0, :b].any() and not out[0, 2 * b:].any()


# ---------------------------------------------------------------- LUT closed forms

def small_matrix(seed, d_in, d_out, block, signs=False):
    g = S.rng(seed)
    m = S.matrix(g, d_in, d_out, block)
    if signs:
        m.signs = S.sign_bits(S.rng(seed, 2), d_in)
    return m


@pytest.mark.parametrize("k", [0, 17, 63])
def test_closed_form_all_indices_equal(k):
    # all indices = k, no signs: y[t, 2p+c] = s[2p+c] C[k][c] sqrt(b) sum_blocks x[t, block start]
    d_in, d_out, b = 64, 8, 16
    m = small_matrix(3, d_in, d_out, b)
    m.stream = O.pack_indices(np.full((d_out // 2) * d_in, k))
    x = S.activations(S.rng(4, 0), 3, d_in)
    y = O.linear_f64(x, m)
    xs = x.astype(np.float64)[:, ::b].sum(axis=1)
    C = m.codebook.astype(np.float64)
    sc = m.scales.astype(np.float64)
    expect = np.stack([sc[o] * C[k][o % 2] * math.sqrt(b) * xs for o in range(d_out)], axis=1)
    assert np.allclose(y, expect, rtol=1e-12, atol=1e-14)


def test_dense_weight_layout_by_hand():
    d_in, d_out = 4, 4
    idx = np.array([[1, 0, 2, 3], [3, 2, 1, 0]])  # idx[p, i]
    C = np.zeros((64, 2), np.float16)
    C[0] = (1, 10)
    C[1] = (2, 20)
    C[2] = (3, 30)
    C[3] = (4, 40)
    sc = np.array([1, 2, 0.5, 4], np.float16)
    W = O.dense_weight(O.pack_indices(idx), C, sc, d_in, d_out)
    expect = np.array([[2, 1, 3, 4],            # channel 0 = pair 0, component 0, scale 1
                       [40, 20, 60, 80],        # channel 1 = pair 0, component 1, scale 2
                       [2, 1.5, 1, 0.5],        # channel 2 = pair 1, component 0, scale 0.5
                       [160, 120, 80, 40]])     # channel 3 = pair 1, component 1, scale 4
    assert np.array_equal(W, expect)


def test_dense_weight_product_exact():
    m = small_matrix(5, 64, 64, 64)
    W = O.dense_weight(m.stream, m.codebook, m.scales, 64, 64)
    W32 = O.dense_weight(m.stream, m.codebook, m.scales, 64, 64, apply_scale=False).astype(np.float32) \
        * m.scales.astype(np.float32)[:, None]
    assert np.array_equal(W, W32.astype(np.float64))  # FP16 x FP16 is exact in FP32


def test_codebook_permutation_invariance():
    # normalising LUT order (a permutation of codebook entries with remapped indices)
    # leaves the weights and outputs unchanged
    d_in, d_out, b = 128, 64, 64
    m = small_matrix(6, d_in, d_out, b)
    perm = np.random.default_rng(1).permutation(64)
    idx = O.index_matrix(m.stream, d_in, d_out)
    inv = np.argsort(perm)
    m2 = S.Matrix(d_in, d_out, b, m.codebook[perm], O.pack_indices(inv[idx]), m.scales)
    assert np.array_equal(O.dense_weight(m.stream, m.codebook, m.scales, d_in, d_out),
                          O.dense_weight(m2.stream, m2.codebook, m2.scales, d_in, d_out))
    x = S.activations(S.rng(1, 0), 4, d_in)
    assert np.array_equal(O.linear(x, m), O.linear(x, m2))


def test_linearity_and_zero():
    m = small_matrix(8, 128, 64, 128)
    g = np.random.default_rng(2)
    x1 = g.standard_normal((2, 128))
    x2 = g.standard_normal((2, 128))
    a, b = 0.5, -1.25
    # linear_f64 rounds inputs to FP16, so check linearity on exactly representable inputs
    x1 = (np.round(x1 * 64) / 64).astype(np.float16)
    x2 = (np.round(x2 * 64) / 64).astype(np.float16)
    comb = (a * x1.astype(np.float64) + b * x2.astype(np.float64))
    assert np.array_equal(comb.astype(np.float16).astype(np.float64), comb)
    lhs = O.linear_f64(comb, m)
    rhs = a * O.linear_f64(x1, m) + b * O.linear_f64(x2, m)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    blk = S.mlp_block(S.rng(9), 64, 128, 64)
    assert not O.mlp_f64(np.zeros((3, 64)), blk).any()


# ---------------------------------------------------------------- SiLU

def test_silu_special_points():
    assert O.silu(np.array([0.0]))[0] == 0.0
    xs = np.array([-30.0, -3.0, -0.5, 0.25, 1.0, 4.0, 30.0])
    for x, v in zip(xs, O.silu(xs)):
        assert v == pytest.approx(x / (1 + math.exp(-x)), rel=1e-15)
        # the pages' tanh form
        # (the tanh form cancels for large negative x, hence the absolute slack)
        assert v == pytest.approx(0.5 * x * (1 + math.tanh(x / 2)), rel=1e-12, abs=1e-14)
    # odd-part identity: silu(x) - silu(-x) = x
    assert np.allclose(O.silu(xs) - O.silu(-xs), xs, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("d_in,d_out,T,block,signs", [
    (2, 2, 1, 2, False), (4, 2, 2, 4, False), (8, 4, 3, 4, True), (8, 4, 2, 8, True), (4, 4, 3, 2, False)])
def test_bruteforce_linear(d_in, d_out, T, block, signs):
    m = small_matrix(10 + d_in, d_in, d_out, block, signs)
    x = S.activations(S.rng(11, 0), T, d_in)
    got = O.linear_f64(x, m)
    ref = bf.linear(x.tolist(), m)
    assert np.allclose(got, np.array(ref), rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("d,inter,T,block,signs", [(2, 4, 1, 2, False), (4, 8, 2, 4, True), (8, 4, 3, 2, True)])
def test_bruteforce_mlp(d, inter, T, block, signs):
    blk = S.mlp_block(S.rng(20 + d), d, inter, block)
    if signs:
        S.add_signs(S.rng(20 + d, 2), blk)
    x = S.activations(S.rng(21, 0), T, d)
    got = O.mlp_f64(x, blk)
    ref = bf.mlp(x.tolist(), blk)
    assert np.allclose(got, np.array(ref), rtol=1e-10, atol=1e-15)


def test_stack_matches_layerwise_definition():
    wl = S.mlp_stack(seed=5, rows=3, layers=3, hidden=64, inter=128, block=64)
    trace = []
    r = O.stack(wl.x, wl.layers, trace=trace)
    assert len(trace) == 4 and np.array_equal(trace[-1], r)
    rr = wl.x.astype(np.float16)
    for blk in wl.layers:
        n = rr.astype(np.float64)
        n = (n / np.sqrt((n * n).mean(axis=1, keepdims=True) + 1e-6)).astype(np.float16)
        y = np.array(bf.mlp(n.tolist(), blk)).astype(np.float16)
        rr = (rr.astype(np.float64) + y.astype(np.float64)).astype(np.float16)
    assert np.array_equal(rr, r)


def test_threaded_ranges_and_generator_blocks_match():
    # output channels in several ranges on several threads: the same values as one serial
    # pass, and as the brute force; a stack fed a generator equals one fed a list
    m = small_matrix(40, 8, 16, 4, True)
    x = S.activations(S.rng(41, 0), 3, 8)
    serial = O.linear_f64(x, m)
    threaded = O.linear_f64(x, m, row_chunk=4, workers=3)
    assert np.array_equal(serial, threaded)
    assert np.allclose(threaded, np.array(bf.linear(x.tolist(), m)), rtol=1e-12, atol=1e-15)
    wl = S.mlp_stack(seed=6, rows=2, layers=3, hidden=64, inter=128, block=64)
    ref = O.stack(wl.x, wl.layers)
    assert np.array_equal(O.stack(wl.x, (b for b in wl.layers), workers=2), ref)


def test_rmsnorm_unit_rms():
    x = S.activations(S.rng(3, 0), 4, 512) * np.float16(3)
    n = O.rmsnorm(x).astype(np.float64)
    assert np.allclose(np.sqrt((n * n).mean(axis=1)), 1.0, atol=2e-3)


# ---------------------------------------------------------------- metrics

def test_metrics():
    ref = np.array([[1.0, -2.0, 4.0]])
    assert O.rel_max_err(ref, ref) == 0.0
    assert O.rel_max_err(ref + np.array([[0, 0, 0.004]]), ref) == pytest.approx(1e-3)
    assert O.row_cosine(ref, ref)[0] == pytest.approx(1.0)
    assert O.row_cosine(ref, -ref)[0] == pytest.approx(-1.0)


# ---------------------------------------------------------------- planted mistakes

def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible oracle bugs (on the CPU) and show a pin fails for each."""
    # 1. MSB-first bit order breaks the golden packing example
    def unpack_msb(stream, start, count):
        bits = np.unpackbits(np.asarray(stream, np.uint8), bitorder="big")[6 * start: 6 * (start + count)]
        return bits.reshape(count, 6).astype(np.int64) @ (np.int64(1) << np.arange(6))
    _, idx, byts = load_pack_golden()[0]
    assert unpack_msb(np.frombuffer(byts, np.uint8), 0, len(idx)).tolist() != idx

    # 2. a dropped 1/sqrt(b) breaks the double-rotation identity
    x = np.random.default_rng(0).standard_normal((1, 16))
    monkeypatch.setattr(O, "rotation_block", lambda b, s=None: O.hadamard(b) * (1 if s is None else s[None, :]))
    assert not np.allclose(O.rotate(O.rotate(x, 16), 16), x)
    monkeypatch.undo()

    # 3. swapped centroid components break the hand-made dense-weight check
    idx = np.array([[1, 0, 2, 3], [3, 2, 1, 0]])
    C = np.zeros((64, 2), np.float16)
    C[:4] = [(1, 10), (2, 20), (3, 30), (4, 40)]
    sc = np.ones(4, np.float16)
    W = O.dense_weight(O.pack_indices(idx), C, sc, 4, 4)
    W_bad = O.dense_weight(O.pack_indices(idx), C[:, ::-1], sc, 4, 4)
    assert W[0, 0] == 2 and W_bad[0, 0] != 2

    # 4. a sign error in SiLU breaks the special points (the odd-part identity alone
    #    would not catch it: z/(1+exp(z)) satisfies it too, so the pin also checks values)
    bad = lambda z: z / (1.0 + np.exp(z))
    assert bad(np.array([1.0]))[0] != pytest.approx(1.0 / (1 + math.exp(-1.0)), rel=1e-6)

    # 5. a transposed weight (W instead of W^T) is caught by the brute force on a non-square case
    m = small_matrix(30, 8, 4, 4)
    x = S.activations(S.rng(31, 0), 2, 8)
    ref = np.array(bf.linear(x.tolist(), m))
    xr = O.rotate(x.astype(np.float64), 4)
    W = O.dense_weight(m.stream, m.codebook, m.scales, 8, 4)
    assert np.allclose(xr @ W.T, ref, rtol=1e-12)
    Wt = W.reshape(-1)[: 8 * 4].reshape(8, 4)  # wrong orientation reading of the same buffer
    assert not np.allclose(xr @ Wt, ref)
