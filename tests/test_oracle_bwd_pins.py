"""Pins for the oracle's backward pass: every gradient against central finite
differences of a weighted loss through the forward oracle, plus the alpha == 1
closed forms.  No GPU needed."""
import numpy as np
import pytest

import oracle


def _inputs(seed, L=7, dk=3, dv=2, BH=1, gate=True):
    r = np.random.default_rng(seed)
    q, k = r.standard_normal((BH, L, dk)), r.standard_normal((BH, L, dk))
    v = r.standard_normal((BH, L, dv))
    la = r.uniform(-0.6, -0.05, (BH, L, dk)) if gate else None
    s0 = r.standard_normal((BH, dk, dv)) * 0.5
    Wo, Wf = r.standard_normal((BH, L, dv)), r.standard_normal((BH, dk, dv))
    return q, k, v, la, s0, Wo, Wf


def _loss(q, k, v, la, s0, Wo, Wf):
    out, fs, _ = oracle.gla_fwd(q, k, v, la, init_state=s0)
    return float(np.sum(out * Wo) + np.sum(fs * Wf))


def _fd(fn, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = fn()
        x[i] = old - h
        fm = fn()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("gate", [True, False])
def test_gradients_match_finite_differences(gate):
    q, k, v, la, s0, Wo, Wf = _inputs(1, gate=gate)
    dq, dk, dv, dla, ds0 = oracle.gla_bwd(q, k, v, Wo, la, s0, Wf)
    f = lambda: _loss(q, k, v, la, s0, Wo, Wf)
    for name, got, x in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v), ("dinit", ds0, s0)) + \
            ((("dlog_alpha", dla, la),) if gate else ()):
        ref = _fd(f, x)
        assert np.max(np.abs(got - ref)) <= 1e-6 * max(1.0, np.max(np.abs(ref))), name


def test_no_final_gradient_and_no_init():
    q, k, v, la, _, Wo, _ = _inputs(2, L=5, dk=2, dv=3)
    dq, dk, dv, dla, ds0 = oracle.gla_bwd(q, k, v, Wo, la, None, None)
    f = lambda: float(np.sum(oracle.gla_fwd(q, k, v, la)[0] * Wo))
    assert np.max(np.abs(dla - _fd(f, la))) <= 1e-6 * max(1.0, np.max(np.abs(dla)))
    assert np.max(np.abs(dv - _fd(f, v))) <= 1e-6 * max(1.0, np.max(np.abs(dv)))


def test_alpha_one_closed_forms():
    """alpha == 1, no initial or final state: dv_t = sum_{s>=t} (q_s.k_t) do_s,
    dq_t = sum_{i<=t} (do_t.v_i) k_i, dk_t = sum_{s>=t} (do_s.v_t) q_s."""
    r = np.random.default_rng(3)
    L, dk, dv = 9, 4, 3
    q, k, v, do = (r.standard_normal((1, L, d)) for d in (dk, dk, dv, dv))
    dq, dkk, dvv, _, _ = oracle.gla_bwd(q, k, v, do)
    M = np.tril(np.ones((L, L)))
    A = q[0] @ k[0].T * M                      # A[t, i] = q_t.k_i for i <= t
    B = do[0] @ v[0].T * M                     # B[t, i] = do_t.v_i for i <= t
    assert np.allclose(dvv[0], A.T @ do[0], atol=1e-12)
    assert np.allclose(dq[0], B @ k[0], atol=1e-12)
    assert np.allclose(dkk[0], B.T @ q[0], atol=1e-12)


def test_two_token_scalar_worked_by_hand():
    """dk = dv = 1, L = 2, no initial state: the loss o_0 + o_1 with
    o_0 = q_0 k_0 v_0 and o_1 = q_1 (a_1 k_0 v_0 + k_1 v_1), differentiated by hand.
    q = (1, 2), k = (3, 1), v = (2, -1), a = (1/2, 1/2):
    dq = (6, 2), dk = (q_0 v_0 + q_1 a_1 v_0, q_1 v_1) = (4, -2),
    dv = (q_0 k_0 + q_1 a_1 k_0, q_1 k_1) = (6, 2),
    dlog a = (0, a_1 q_1 k_0 v_0) = (0, 6), dS_init = a_0 (q_0 + q_1 a_1) = 1."""
    q = np.array([[[1.0], [2.0]]])
    k = np.array([[[3.0], [1.0]]])
    v = np.array([[[2.0], [-1.0]]])
    la = np.log(np.full((1, 2, 1), 0.5))
    dq, dk, dv, dla, ds0 = oracle.gla_bwd(q, k, v, np.ones((1, 2, 1)), la, np.zeros((1, 1, 1)))
    assert np.allclose(dq.ravel(), [6, 2], atol=1e-14)
    assert np.allclose(dk.ravel(), [4, -2], atol=1e-14)
    assert np.allclose(dv.ravel(), [6, 2], atol=1e-14)
    assert np.allclose(dla.ravel(), [0, 6], atol=1e-14)
    assert np.allclose(ds0.ravel(), [1], atol=1e-14)


def test_per_token_gate_gradient_is_the_channel_sum():
    """One gate per token shared by all channels (log alpha_t[i] = g_t): by the
    chain rule dL/dg_t is the sum over channels of the per-channel gradient;
    checked against finite differences in g through the forward oracle."""
    q, k, v, _, s0, Wo, Wf = _inputs(6, L=6, dk=3, dv=2)
    g = np.random.default_rng(7).uniform(-0.5, -0.05, (1, 6))
    wide = lambda: np.repeat(g[..., None], 3, axis=-1)
    _, _, _, dla, _ = oracle.gla_bwd(q, k, v, Wo, wide(), s0, Wf)
    f = lambda: _loss(q, k, v, wide(), s0, Wo, Wf)
    ref = _fd(f, g)
    got = dla.sum(axis=-1)
    assert np.max(np.abs(got - ref)) <= 1e-6 * max(1.0, np.max(np.abs(ref)))
