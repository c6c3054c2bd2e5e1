"""Pins for the gated delta-rule oracle (oracle/delta_rule.py): the pages' closed
form of the 8-row block inverse ("anemll/anemll-forge-qwen3.8-27B", "Faster
exact graph (previous update)", bullet "Gated DeltaNet") against nilpotency,
forward substitution and numpy's solver; the recurrence against cases with a
known answer; and the block form a kernel uses against the recurrence."""

import numpy as np
import pytest

from oracle import delta_rule as D
from synth import inputs as S


def strict_lower(g, n=8, scale=1.0):
    return np.tril(g.standard_normal((n, n)) * scale, -1)


@pytest.mark.parametrize("seed", range(5))
def test_block_inverse_closed_form(seed):
    g = np.random.default_rng(seed)
    N = strict_lower(g, 8, 0.7)
    assert np.array_equal(np.linalg.matrix_power(N, 8), np.zeros((8, 8)))  # nilpotent, exactly
    P = D.block_solve(N)
    eye = np.eye(8)
    assert np.allclose(P @ (eye + N), eye, atol=1e-12)
    assert np.allclose(P, D.triangular_inverse(N), atol=1e-12)
    assert np.allclose(P, np.linalg.inv(eye + N), atol=1e-10)


def test_block_inverse_by_hand():
    # N = a e_1 e_0^T: (I + N)^-1 = I - N
    N = np.zeros((8, 8))
    N[1, 0] = 3.0
    expect = np.eye(8)
    expect[1, 0] = -3.0
    assert np.array_equal(D.block_solve(N), expect)


def test_single_token_by_hand():
    # S1 = a S0 + b k (v - a S0^T k)^T, o = S1^T q
    S0 = np.array([[1.0], [2.0]])
    k = np.array([[1.0, 0.0]])
    v = np.array([[5.0]])
    out, S1 = D.recurrent(np.array([[0.0, 1.0]]), k, v, np.array([0.5]), np.array([0.5]), S0)
    # a S0^T k = 0.5; u = 4.5; S1 = [[0.5], [1.0]] + 0.5 [1, 0]^T 4.5 = [[2.75], [1.0]]
    assert np.array_equal(S1, np.array([[2.75], [1.0]]))
    assert np.array_equal(out, np.array([[1.0]]))


def test_zero_strength_only_decays():
    g = np.random.default_rng(1)
    T, dk, dv = 8, 6, 5
    q, k, v = g.standard_normal((T, dk)), g.standard_normal((T, dk)), g.standard_normal((T, dv))
    alpha = g.uniform(0.8, 1.0, T)
    S0 = g.standard_normal((dk, dv))
    out, S = D.recurrent(q, k, v, np.zeros(T), alpha, S0)
    gam = np.cumprod(alpha)
    assert np.allclose(S, gam[-1] * S0, atol=1e-13)
    assert np.allclose(out, gam[:, None] * (q @ S0), atol=1e-12)


def test_orthonormal_keys_store_exactly():
    # unit strength and gate, orthonormal keys, empty state: the state is an exact
    # associative memory, S^T k_j = v_j, and a repeated key overwrites (delta rule)
    T, dk, dv = 8, 8, 3
    k = np.eye(dk)[:T]
    v = np.arange(T * dv, dtype=np.float64).reshape(T, dv)
    _, S = D.recurrent(k, k, v, np.ones(T), np.ones(T), np.zeros((dk, dv)))
    assert np.allclose(k @ S, v, atol=1e-13)
    k2 = np.stack([k[0], k[0]])
    _, S2 = D.recurrent(k2, k2, np.array([[1.0, 2, 3], [7.0, 8, 9]]), np.ones(2), np.ones(2), np.zeros((dk, dv)))
    assert np.allclose(S2.T @ k[0], [7, 8, 9], atol=1e-13)


def block_form(q, k, v, beta, alpha, S0):
    """The 8-row block as a kernel computes it (derivation written out):
    gamma_t = prod_{s<=t} alpha_s; N[t, j] = (gamma_t / gamma_j) beta_j k_t.k_j (j < t);
    U = (I + N)^-1 (V - Gamma K S0); O = Gamma Q S0 + M U with M[t, j] = (gamma_t /
    gamma_j) beta_j q_t.k_j (j <= t); S = gamma_T S0 + K^T diag(beta_j gamma_T / gamma_j) U."""
    gam = np.cumprod(alpha)
    ratio = gam[:, None] / gam[None, :]
    N = np.tril(ratio * (k @ k.T) * beta[None, :], -1)
    U = D.block_solve(N) @ (v - gam[:, None] * (k @ S0))
    M = np.tril(ratio * (q @ k.T) * beta[None, :])
    out = gam[:, None] * (q @ S0) + M @ U
    S = gam[-1] * S0 + k.T @ ((beta * gam[-1] / gam)[:, None] * U)
    return out, S


@pytest.mark.parametrize("seed", range(4))
def test_block_form_equals_recurrence(seed):
    g = np.random.default_rng(seed)
    T, dk, dv = 8, 16, 12
    q = g.standard_normal((T, dk))
    k = g.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = g.standard_normal((T, dv))
    beta = g.uniform(0.05, 0.95, T)
    alpha = g.uniform(0.85, 1.0, T)
    S0 = g.standard_normal((dk, dv)) * 0.3
    o1, s1 = D.recurrent(q, k, v, beta, alpha, S0)
    o2, s2 = block_form(q, k, v, beta, alpha, S0)
    assert np.allclose(o1, o2, atol=1e-11) and np.allclose(s1, s2, atol=1e-11)


def test_planted_mistake_in_the_inverse_is_caught():
    # dropping the last factor (I + N^4) gives only the first four terms of the series
    g = np.random.default_rng(9)
    N = strict_lower(g, 8, 0.7)
    eye = np.eye(8)
    wrong = (eye - N) @ (eye + N @ N)
    assert not np.allclose(wrong, D.triangular_inverse(N), atol=1e-6)


def test_generator_shapes():
    w = S.delta_rule_inputs(seed=7, tokens=16, heads=2, d_k=32, d_v=16)
    assert w.q.shape == (16, 2, 32) and w.v.shape == (16, 2, 16) and w.state.shape == (2, 32, 16)
    assert np.allclose(np.linalg.norm(w.k.astype(np.float64), axis=-1), 1.0, atol=2e-3)
