"""CPU oracle for the gated delta-rule token mixer, one head at a time.

TEST INFRASTRUCTURE ONLY (like oracle/vq3_oracle.py): only the tests, the
entry point's smoke check and the benchmark's CPU baseline use it; it shares no
code with the CUDA library.

Source: "anemll/anemll-forge-qwen3.8-27B", section "Faster exact graph
(previous update)", bullet "Gated DeltaNet": verification and prefill process
tokens in 8-row blocks; every token's delta-rule update depends on the earlier
tokens of its block, a triangular solve, whose exact closed form for the
strictly lower-triangular block N is (I + N)^-1 = (I - N)(I + N^2)(I + N^4).

The pages name the gated delta rule without writing it out. The plainest
reading, taken here: a head keeps a state S [d_k, d_v]; token t (query q_t, key
k_t, value v_t, strength beta_t, gate alpha_t) updates it and reads it out as

    S_t = alpha_t S_{t-1} + beta_t k_t (v_t - alpha_t S_{t-1}^T k_t)^T
    o_t = S_t^T q_t

This module computes exactly that, token by token, in float64 (`recurrent`).
`block_solve` writes out the pages' closed form of the block inverse, and
`triangular_inverse` the plain row-by-row forward substitution it replaces;
the tests pin one against the other and against numpy's solver.
"""

from __future__ import annotations

import numpy as np


def recurrent(q, k, v, beta, alpha, state):
    """Outputs [T, d_v] and the final state, token by token, float64.

    q, k: [T, d_k]; v: [T, d_v]; beta, alpha: [T]; state: [d_k, d_v].
    """
    S = np.array(state, dtype=np.float64)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    beta = np.asarray(beta, np.float64)
    alpha = np.asarray(alpha, np.float64)
    out = np.empty((q.shape[0], v.shape[1]), dtype=np.float64)
    for t in range(q.shape[0]):
        u = v[t] - alpha[t] * (S.T @ k[t])           # the delta-rule "new value"
        S = alpha[t] * S + beta[t] * np.outer(k[t], u)
        out[t] = S.T @ q[t]
    return out, S


def block_solve(N):
    """(I + N)^-1 for a strictly lower-triangular 8 x 8 block, as the pages write
    it: (I - N)(I + N^2)(I + N^4) (exact because N^8 = 0)."""
    N = np.asarray(N, np.float64)
    eye = np.eye(N.shape[0])
    N2 = N @ N
    N4 = N2 @ N2
    return (eye - N) @ (eye + N2) @ (eye + N4)


def triangular_inverse(N):
    """(I + N)^-1 by forward substitution, one row after another (the solve the
    closed form replaces)."""
    N = np.asarray(N, np.float64)
    n = N.shape[0]
    X = np.zeros((n, n))
    for i in range(n):
        row = np.zeros(n)
        row[i] = 1.0
        for j in range(i):
            row -= N[i, j] * X[j]
        X[i] = row
    return X
