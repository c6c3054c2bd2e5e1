"""Pins for the oracle's low-rank correction: W = diag(s) C[idx] + U V, the
factors acting on the rotated input like the lookup-table part (model card
"anemll/anemll-forge-qwen3.8-27B", release-comparison table row "Token mixers":
rank-64 factors; "ANEMLL ANE LLM conversion pipeline", "Facts": rank-64
residual correction). Checked against a closed form that uses the rotation's
orthogonality and against the pure-Python brute force."""

import numpy as np
import pytest

from oracle import bruteforce as bf
from oracle import vq3_oracle as O
from synth import inputs as S


@pytest.mark.parametrize("fmt", ["2x64", "2x16", "lut4"])
@pytest.mark.parametrize("d_in,d_out,T,block,rank", [(4, 2, 2, 4, 1), (8, 4, 3, 4, 3), (8, 8, 2, 8, 2)])
def test_bruteforce_linear_with_factors(fmt, d_in, d_out, T, block, rank):
    m = S.matrix(S.rng(60 + d_in), d_in, d_out, block, fmt)
    m.signs = S.sign_bits(S.rng(60 + d_in, 2), d_in)
    S.add_lowrank(S.rng(60 + d_in, 3), m, rank, 0.3)
    x = S.activations(S.rng(61, 0), T, d_in)
    assert np.allclose(O.linear_f64(x, m), np.array(bf.linear(x.tolist(), m)), rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("rank", [1, 4, 16])
def test_closed_form_factor_undoes_the_rotation(rank):
    # With a zero codebook the lookup-table part vanishes. Choosing V's rows as
    # columns of the rotation (V[j][i] = R[i][j]) gives V x' = V R x = x[:rank]
    # (R is orthogonal), so y = U x[:, :rank]^T whatever the scales are.
    d_in, d_out, b = 64, 8, 16
    m = S.matrix(S.rng(62), d_in, d_out, b)
    m.codebook = np.zeros_like(m.codebook)
    R = O.rotation_block(b)  # entries +-1/4: exact in FP16
    V = np.zeros((rank, d_in))
    V[:, :b] = R[:, :rank].T
    m.lr_v = V.astype(np.float16)
    m.lr_u = (np.random.default_rng(5).standard_normal((d_out, rank)) * 0.5).astype(np.float16)
    x = S.activations(S.rng(63, 0), 3, d_in)
    expect = x.astype(np.float64)[:, :rank] @ m.lr_u.astype(np.float64).T
    assert np.allclose(O.linear_f64(x, m), expect, rtol=1e-12, atol=1e-12)


def test_zero_factors_change_nothing():
    m = S.matrix(S.rng(64), 128, 64, 64, "2x16")
    x = S.activations(S.rng(64, 0), 4, 128)
    y0 = O.linear_f64(x, m)
    m.lr_u = np.zeros((64, 8), np.float16)
    m.lr_v = np.zeros((8, 128), np.float16)
    assert np.array_equal(O.linear_f64(x, m), y0)


def test_planted_mistake_scaling_the_factors_is_caught():
    # scaling the correction by the per-channel scales (a plausible slip) breaks the closed form
    d_in, d_out, b, rank = 64, 8, 16, 4
    m = S.matrix(S.rng(65), d_in, d_out, b)
    m.codebook = np.zeros_like(m.codebook)
    R = O.rotation_block(b)
    V = np.zeros((rank, d_in))
    V[:, :b] = R[:, :rank].T
    m.lr_v = V.astype(np.float16)
    m.lr_u = np.ones((d_out, rank), np.float16)
    x = S.activations(S.rng(66, 0), 2, d_in)
    good = O.linear_f64(x, m)
    wrong = good * m.scales.astype(np.float64)[None, :]
    expect = x.astype(np.float64)[:, :rank] @ m.lr_u.astype(np.float64).T
    assert np.allclose(good, expect) and not np.allclose(wrong, expect)
