"""The chunked form of the gated delta rule that dn_prefill's recurrence
kernels evaluate (on the CUDA cores and on the tensor cores: chunks of up to
32 tokens of one value head with one decay per head), checked on the CPU in
float64 against the oracle stepping the same tokens one by one.

For a chunk with state S0 at its start, cumulative log-decays
G_t = g_0 + ... + g_t and gamma_t = exp(G_t), substituting the token
recurrence into itself gives

    u_t = beta_t (v_t - gamma_t S0^T k_t - sum_{s<t} exp(G_t - G_s) (k_t.k_s) u_s)
    o_t = gamma_t S0^T q_t + sum_{s<=t} exp(G_t - G_s) (q_t.k_s) u_s
    S   = gamma_n S0 + sum_t exp(G_n - G_t) k_t u_t^T

(u_t is the token's delta against its decayed state).  The kernels compute
these sums in other orders and precisions; this test pins the algebra
itself, so a sign, an exponent or a strict-versus-inclusive bound taken
wrongly in the derivation fails here without a GPU."""
import numpy as np
import pytest

from oracle import gated_delta_rule_step


def chunk_form(S0, Q, K, V, g, beta):
    """The chunk's final state and its readouts, from the closed forms above."""
    n = len(g)
    G = np.cumsum(g)
    gam = np.exp(G)
    U = np.zeros_like(V)
    for t in range(n):
        acc = V[t] - gam[t] * (S0.T @ K[t])
        for s in range(t):
            acc = acc - np.exp(G[t] - G[s]) * (K[t] @ K[s]) * U[s]
        U[t] = beta[t] * acc
    O = np.zeros_like(V)
    for t in range(n):
        O[t] = gam[t] * (S0.T @ Q[t])
        for s in range(t + 1):
            O[t] = O[t] + np.exp(G[t] - G[s]) * (Q[t] @ K[s]) * U[s]
    S = gam[n - 1] * S0
    for t in range(n):
        S = S + np.exp(G[n - 1] - G[t]) * np.outer(K[t], U[t])
    return S, O


def serial(S0, Q, K, V, g, beta):
    S, O = S0, np.zeros_like(V)
    for t in range(len(g)):
        S, O[t] = gated_delta_rule_step(S, Q[t], K[t], V[t], g[t], beta[t])
    return S, O


def random_chunk(rng, n, dk=8, dv=6):
    K = rng.standard_normal((n, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)  # the kernels take L2-normalised keys
    Q = rng.standard_normal((n, dk)) / np.sqrt(dk)
    V = rng.standard_normal((n, dv))
    g = -rng.uniform(0.0, 0.7, n)
    beta = rng.uniform(0.05, 1.0, n)
    return Q, K, V, g, beta


@pytest.mark.parametrize("n", [1, 2, 5, 32])
def test_chunk_form_equals_token_steps(n):
    rng = np.random.default_rng(100 + n)
    S0 = rng.standard_normal((8, 6)) * 0.3
    Q, K, V, g, beta = random_chunk(rng, n)
    S_c, O_c = chunk_form(S0, Q, K, V, g, beta)
    S_s, O_s = serial(S0, Q, K, V, g, beta)
    np.testing.assert_allclose(S_c, S_s, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(O_c, O_s, rtol=1e-11, atol=1e-12)


def test_chunks_chain_like_the_token_recurrence():
    """70 tokens as chunks of 32, 32 and 6 (a ragged last chunk), each
    starting from the state the previous one ends with."""
    rng = np.random.default_rng(7)
    S0 = rng.standard_normal((8, 6)) * 0.3
    Q, K, V, g, beta = random_chunk(rng, 70)
    S, outs = S0, []
    for c0, c1 in ((0, 32), (32, 64), (64, 70)):
        S, O = chunk_form(S, Q[c0:c1], K[c0:c1], V[c0:c1], g[c0:c1], beta[c0:c1])
        outs.append(O)
    S_s, O_s = serial(S0, Q, K, V, g, beta)
    np.testing.assert_allclose(S, S_s, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(outs), O_s, rtol=1e-10, atol=1e-12)


def test_zero_write_strength_leaves_pure_decay():
    """beta = 0: every delta is zero, the state only decays (gamma_n S0) and
    the readouts are gamma_t S0^T q_t."""
    rng = np.random.default_rng(3)
    S0 = rng.standard_normal((8, 6))
    Q, K, V, g, _ = random_chunk(rng, 9)
    S, O = chunk_form(S0, Q, K, V, g, np.zeros(9))
    G = np.cumsum(g)
    np.testing.assert_allclose(S, np.exp(G[-1]) * S0, rtol=1e-13)
    np.testing.assert_allclose(O, np.exp(G)[:, None] * (Q @ S0), rtol=1e-13)
