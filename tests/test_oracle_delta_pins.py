"""Pins for the oracle's delta rule ("linear-attention" blog, Delta attention):
checked against the pages' own triangular-system form of prefill (solved with
a library routine), exact retrieval with orthonormal keys, the beta = 0 case
and a hand-worked example.  No GPU needed."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _close(a, b, rtol=1e-10):
    a, b = np.asarray(a, float), np.asarray(b, float)
    return float(np.max(np.abs(a - b))) <= rtol * max(1.0, float(np.max(np.abs(b))))


def _inputs(seed, L, dk, dv, BH=2, unit_keys=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((BH, L, dk))
    k = r.standard_normal((BH, L, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((BH, L, dv))
    beta = r.uniform(0.05, 0.95, (BH, L))
    return q, k, v, beta


def triangular_form(q, k, v, beta, s0, gamma=None):
    """Prefill as one lower-triangular system (the pages' derivation): the writes u_n
    satisfy u_n + beta_n sum_{i<n} G[n,i] (k_n . k_i) u_i = beta_n (v_n - G[n,-1] S0^T k_n),
    with G[n,i] the product of the per-token decays over (i, n] (all ones without a gate).
    Then o_n = G[n,-1] S0^T q_n + sum_{i<=n} G[n,i] (q_n . k_i) u_i."""
    L = q.shape[0]
    lg = np.zeros(L) if gamma is None else np.log(gamma)
    c = np.cumsum(lg)
    G = np.exp(c[:, None] - c[None, :])          # G[n, i] = prod over (i, n]
    g0 = np.exp(c)                               # decay of S0 up to n (inclusive)
    Mk = np.tril(k @ k.T * G, -1)
    A = np.eye(L) + beta[:, None] * Mk
    rhs = beta[:, None] * (v - g0[:, None] * (k @ s0))
    U = np.linalg.solve(A, rhs)
    O = g0[:, None] * (q @ s0) + np.tril(q @ k.T * G) @ U
    S = g0[-1] * s0 + (k * G[-1][:, None]).T @ U
    return O, S


def test_triangular_system_equals_recurrence():
    q, k, v, beta = _inputs(1, 40, 6, 5)
    s0 = np.random.default_rng(11).standard_normal((2, 6, 5)) * 0.3
    out, fs = oracle.delta_fwd(q, k, v, beta, init_state=s0)
    for h in range(2):
        O, S = triangular_form(q[h], k[h], v[h], beta[h], s0[h])
        assert _close(out[h], O) and _close(fs[h], S)


def test_triangular_system_with_per_token_decay():
    q, k, v, beta = _inputs(2, 30, 4, 3)
    gamma = np.random.default_rng(12).uniform(0.6, 0.99, (2, 30))
    s0 = np.random.default_rng(13).standard_normal((2, 4, 3)) * 0.3
    la = np.repeat(np.log(gamma)[..., None], 4, axis=-1)   # the same decay on every channel
    out, fs = oracle.delta_fwd(q, k, v, beta, log_alpha=la, init_state=s0)
    for h in range(2):
        O, S = triangular_form(q[h], k[h], v[h], beta[h], s0[h], gamma[h])
        assert _close(out[h], O) and _close(fs[h], S)


def test_orthonormal_keys_are_retrieved_exactly():
    """beta = 1 and orthonormal keys: each write replaces what the memory held for that key,
    so the final state returns every written value, whatever the initial state."""
    r = np.random.default_rng(3)
    dk, dv, L = 8, 5, 6
    K = np.linalg.qr(r.standard_normal((dk, dk)))[0][:, :L].T      # L orthonormal rows
    v = r.standard_normal((1, L, dv))
    s0 = r.standard_normal((1, dk, dv))
    _, fs = oracle.delta_fwd(r.standard_normal((1, L, dk)), K[None], v, np.ones((1, L)), init_state=s0)
    assert _close(K @ fs[0], v[0], 1e-12)


def test_beta_zero_keeps_the_state():
    q, k, v, _ = _inputs(4, 12, 4, 3)
    s0 = np.random.default_rng(14).standard_normal((2, 4, 3))
    la = np.log(np.random.default_rng(15).uniform(0.5, 1.0, (2, 12, 4)))
    out, fs = oracle.delta_fwd(q, k, v, np.zeros((2, 12)), log_alpha=la, init_state=s0)
    dec = np.exp(np.cumsum(la, axis=1))          # [BH, L, dk]: decay of S0's rows up to t
    assert _close(out, np.einsum("btd,btd,bdj->btj", q, dec, s0))
    assert _close(fs, dec[:, -1][..., None] * s0)


def test_golden_hand_worked():
    with open(os.path.join(GOLDEN, "delta_2x2.json")) as f:
        g = json.load(f)
    q, k, v = (np.array(g[n], float)[None] for n in ("q", "k", "v"))
    b = np.array(g["beta"], float)[None]
    out, fs = oracle.delta_fwd(q, k, v, b)
    assert _close(out[0], g["expect_out"], 1e-14) and _close(fs[0], g["expect_final_state"], 1e-14)
    la = np.log(np.array(g["gated_alpha"], float))[None]
    out, fs = oracle.delta_fwd(q, k, v, b, log_alpha=la)
    assert _close(out[0], g["gated_expect_out"], 1e-14) and _close(fs[0], g["gated_expect_final_state"], 1e-14)
