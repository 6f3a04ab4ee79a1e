"""Pins for the fp64 oracle against facts the pages fix (no GPU needed).

Every pin here checks the oracle against something other than itself: a
closed form, a brute-force evaluation of a different form of the method, an
identity stated on the pages, or a hand-derived worked example.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RTOL = 1e-11


def _rng(seed):
    return np.random.default_rng(seed)


def _inputs(seed, L, dk, dv, BH=2, gate=True, lo=-0.5, hi=-0.001):
    r = _rng(seed)
    q = r.standard_normal((BH, L, dk))
    k = r.standard_normal((BH, L, dk))
    v = r.standard_normal((BH, L, dv))
    la = r.uniform(lo, hi, (BH, L, dk)) if gate else None
    return q, k, v, la


def _close(a, b, rtol=RTOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    return float(np.max(np.abs(a - b))) <= rtol * scale if a.size else True


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


# ---------------------------------------------------------------- brute-force forms

def quadratic_masked(q, k, v, la, s0=None):
    """O[t] = sum_{i<=t} sum_d q[t,d] k[i,d] exp(B[t,d]-B[i,d]) v[i] (+ init term).

    B is the inclusive cumulative sum of log alpha over the whole sequence:
    a write at i survives to t with the product of alpha over (i, t].
    """
    BH, L, dk = q.shape
    out = np.zeros((BH, L, v.shape[-1]))
    for bh in range(BH):
        Bc = np.cumsum(la[bh], axis=0) if la is not None else np.zeros((L, dk))
        for t in range(L):
            w = np.exp(Bc[t][None, :] - Bc[: t + 1])          # [i, d]
            a = np.einsum("d,id,id->i", q[bh, t], k[bh, : t + 1], w)
            out[bh, t] = a @ v[bh, : t + 1]
            if s0 is not None:
                out[bh, t] += (q[bh, t] * np.exp(Bc[t])) @ s0[bh]
    return out


# ---------------------------------------------------------------- pins

def test_alpha_one_is_cumsum():
    """alpha == 1: S_t is the running sum of k_i v_i^T (a plain cumsum)."""
    q, k, v, _ = _inputs(1, 37, 5, 3, gate=False)
    out, fs, _ = oracle.gla_fwd(q, k, v)
    outer = np.einsum("bld,blj->bldj", k, v)
    S = np.cumsum(outer, axis=1)
    assert _close(fs, S[:, -1])
    assert _close(out, np.einsum("bld,bldj->blj", q, S))


def test_recurrent_equals_quadratic_masked_form():
    """Recurrence == (Q K^T (.) L_decay) V by brute force, per-channel decay."""
    q, k, v, la = _inputs(2, 64, 6, 4)
    out, _, _ = oracle.gla_fwd(q, k, v, la)
    assert _close(out, quadratic_masked(q, k, v, la))


def test_recurrent_equals_quadratic_with_initial_state():
    q, k, v, la = _inputs(3, 40, 4, 5)
    s0 = _rng(33).standard_normal((2, 4, 5))
    out, _, _ = oracle.gla_fwd(q, k, v, la, init_state=s0)
    assert _close(out, quadratic_masked(q, k, v, la, s0))


def test_noncausal_regrouping():
    """Mask removed, alpha == 1: O = Q (K^T V); the final state is K^T V."""
    q, k, v, _ = _inputs(4, 29, 6, 6, gate=False)
    _, fs, _ = oracle.gla_fwd(q, k, v)
    KtV = np.einsum("bld,blj->bdj", k, v)
    assert _close(fs, KtV)
    # a decode step with no write and no decay reads the state: o = (K^T V)^T q
    z = np.zeros_like(q[:, 0])
    o, _ = oracle.gla_decode_step(q[:, 5], z, np.zeros_like(v[:, 0]), z, fs)
    brute = np.einsum("bd,bid,bij->bj", q[:, 5], k, v)   # sum over ALL i of (q.k_i) v_i
    assert _close(o, brute)


def test_normaliser_bruteforce():
    """phi = elu+1 and normaliser: o_t = sum sim v / sum sim over i <= t."""
    q, k, v, _ = _inputs(5, 50, 4, 3, gate=False)
    out, fs, fz = oracle.gla_fwd(q, k, v, feature_elu1=True, normalize=True)
    pq, pk = _phi(q), _phi(k)
    for bh in range(2):
        sim = pq[bh] @ pk[bh].T
        sim = np.tril(sim)
        ref = (sim @ v[bh]) / sim.sum(axis=1, keepdims=True)
        assert _close(out[bh], ref)
        assert _close(fz[bh], pk[bh].sum(axis=0))
        assert _close(fs[bh], pk[bh].T @ v[bh])


def test_normaliser_with_gate_decays_z():
    """Reading: z is the state's extra all-ones value column, so it decays too."""
    q, k, v, la = _inputs(6, 30, 3, 2)
    out, _, _ = oracle.gla_fwd(q, k, v, la, feature_elu1=True, normalize=True)
    pq, pk = _phi(q), _phi(k)
    ones = np.ones(v.shape[:-1] + (1,))
    num = quadratic_masked(pq, pk, v, la)
    den = quadratic_masked(pq, pk, ones, la)
    assert _close(out, num / den)


def test_normaliser_with_initial_state_and_z_bruteforce():
    """Resuming the normalised form from a given (S_0, z_0): numerator and denominator each
    carry their initial value decayed to t, o_t = phi(q_t)^T (D_t S_0 + sum_i W_ti phi(k_i) v_i^T)
    / phi(q_t)^T (D_t z_0 + sum_i W_ti phi(k_i)), with D_t = e^{B_t} and W_ti = e^{B_t - B_i} per
    channel ("Transformers are RNNs" notes, normalised kernel form; z is the all-ones value
    column of the state, so it decays like S)."""
    q, k, v, la = _inputs(16, 40, 3, 2)
    r = _rng(17)
    s0 = r.standard_normal((2, 3, 2))
    z0 = r.uniform(0.5, 2.0, (2, 3))
    out, fs, fz = oracle.gla_fwd(q, k, v, la, init_state=s0, init_z=z0, feature_elu1=True, normalize=True)
    pq, pk = _phi(q), _phi(k)
    for bh in range(2):
        Bc = np.cumsum(la[bh], axis=0)
        for t in range(40):
            w = np.exp(Bc[t][None, :] - Bc[: t + 1])  # [i, d]
            num = pq[bh, t] @ (np.exp(Bc[t])[:, None] * s0[bh] + (w * pk[bh, : t + 1]).T @ v[bh, : t + 1])
            den = pq[bh, t] @ (np.exp(Bc[t]) * z0[bh] + (w * pk[bh, : t + 1]).sum(axis=0))
            assert _close(out[bh, t], num / den)
        wL = np.exp(Bc[-1][None, :] - Bc)
        assert _close(fz[bh], np.exp(Bc[-1]) * z0[bh] + (wL * pk[bh]).sum(axis=0))
        assert _close(fs[bh], np.exp(Bc[-1])[:, None] * s0[bh] + (wL * pk[bh]).T @ v[bh])


@pytest.mark.parametrize("L1", [64, 29])
def test_normalised_split_resume(L1):
    """The normalised form split anywhere and resumed from the first part's (S, z) equals the
    whole sequence: the pair (S, z) is a sufficient summary of the prefix."""
    q, k, v, la = _inputs(18, 120, 4, 3)
    out, fs, fz = oracle.gla_fwd(q, k, v, la, feature_elu1=True, normalize=True)
    o1, s1, z1 = oracle.gla_fwd(q[:, :L1], k[:, :L1], v[:, :L1], la[:, :L1], feature_elu1=True, normalize=True)
    o2, s2, z2 = oracle.gla_fwd(q[:, L1:], k[:, L1:], v[:, L1:], la[:, L1:], init_state=s1, init_z=z1,
                                feature_elu1=True, normalize=True)
    assert _close(np.concatenate([o1, o2], axis=1), out)
    assert _close(s2, fs) and _close(z2, fz)


def test_decode_equals_prefill():
    q, k, v, la = _inputs(7, 20, 5, 4)
    s0 = _rng(77).standard_normal((2, 5, 4))
    out, fs, _ = oracle.gla_fwd(q, k, v, la, init_state=s0)
    st = s0.copy()
    for t in range(20):
        o, st = oracle.gla_decode_step(q[:, t], k[:, t], v[:, t], la[:, t], st)
        assert _close(o, out[:, t])
    assert _close(st, fs)


@pytest.mark.parametrize("L1", [64, 37])
def test_split_resume(L1):
    q, k, v, la = _inputs(8, 150, 4, 3)
    out, fs, _ = oracle.gla_fwd(q, k, v, la)
    o1, f1, _ = oracle.gla_fwd(q[:, :L1], k[:, :L1], v[:, :L1], la[:, :L1])
    o2, f2, _ = oracle.gla_fwd(q[:, L1:], k[:, L1:], v[:, L1:], la[:, L1:], init_state=f1)
    assert _close(np.concatenate([o1, o2], axis=1), out)
    assert _close(f2, fs)


@pytest.mark.parametrize("L1", [64, 37])
def test_split_from_zero_state_plus_correction(L1):
    """Linearity in the initial state: the second part run from a zero state,
    plus the decayed first-part state read by each query,
    o_t = o'_t + (q_t * e^{B_t})^T S_A and S = Diag(e^{B_end}) S_A + S',
    with B_t the gate's cumulative sum from the split point (inclusive).  This
    is the identity a split of the sequence across independent chains uses."""
    q, k, v, la = _inputs(9, 160, 4, 3)
    s0 = _rng(10).standard_normal((2, 4, 3))
    out, fs, _ = oracle.gla_fwd(q, k, v, la, init_state=s0)
    o1, sa, _ = oracle.gla_fwd(q[:, :L1], k[:, :L1], v[:, :L1], la[:, :L1], init_state=s0)
    o2, sb, _ = oracle.gla_fwd(q[:, L1:], k[:, L1:], v[:, L1:], la[:, L1:])
    B = np.cumsum(la[:, L1:], axis=1)
    corr = np.einsum("btd,bdj->btj", q[:, L1:] * np.exp(B), sa)
    assert _close(np.concatenate([o1, o2 + corr], axis=1), out)
    assert _close(np.exp(B[:, -1])[..., None] * sa + sb, fs)


@pytest.mark.parametrize("C", [1, 16, 64, 100, 200])
def test_chunk_form_equals_recurrence(C):
    """The chunk-wise form is an exact refactoring for every chunk size C."""
    q, k, v, la = _inputs(9, 100, 5, 3)
    s0 = _rng(99).standard_normal((2, 5, 3))
    out, fs, _ = oracle.gla_fwd(q, k, v, la, init_state=s0)
    oc, fc = oracle.gla_fwd_chunked(q, k, v, la, init_state=s0, chunk=C)
    assert _close(oc, out, 1e-10)
    assert _close(fc, fs, 1e-10)


def test_gate_to_zero_keeps_only_current_token():
    """log alpha -> -inf: o_t = (q_t . k_t) v_t (the history is forgotten)."""
    q, k, v, _ = _inputs(10, 12, 4, 3, gate=False)
    la = np.full(q.shape, -1e4)
    s0 = np.ones((2, 4, 3))
    out, fs, _ = oracle.gla_fwd(q, k, v, la, init_state=s0)
    ref = np.einsum("bld,bld->bl", q, k)[..., None] * v
    assert _close(out, ref)
    assert _close(fs, np.einsum("bd,bj->bdj", k[:, -1], v[:, -1]))


def test_scalar_gate_mamba2_special_case():
    """G_t = gamma_t 1 1^T: the decay mask is a scalar per (t, i)."""
    q, k, v, _ = _inputs(11, 33, 4, 3, gate=False)
    g = _rng(111).uniform(-0.3, -0.01, (2, 33))
    la = np.repeat(g[..., None], 4, axis=-1)
    out, _, _ = oracle.gla_fwd(q, k, v, la)
    for bh in range(2):
        c = np.cumsum(g[bh])
        D = np.tril(np.exp(c[:, None] - c[None, :]))
        ref = ((q[bh] @ k[bh].T) * D) @ v[bh]
        assert _close(out[bh], ref)


def test_constant_decay_retnet_special_case():
    """Constant per-channel alpha: weight alpha_d^(t-i) for a write at i read at t."""
    q, k, v, _ = _inputs(12, 25, 3, 2, gate=False)
    a = np.array([0.9, 0.5, 0.99])
    la = np.broadcast_to(np.log(a), q.shape).copy()
    out, _, _ = oracle.gla_fwd(q, k, v, la)
    for bh in range(2):
        for t in range(25):
            acc = np.zeros(2)
            for i in range(t + 1):
                acc += np.sum(q[bh, t] * k[bh, i] * a ** (t - i)) * v[bh, i]
            assert _close(out[bh, t], acc)


def test_value_columns_are_independent():
    q, k, v, la = _inputs(13, 70, 4, 6)
    out, fs, _ = oracle.gla_fwd(q, k, v, la)
    oa, fa, _ = oracle.gla_fwd(q, k, v[..., :2], la)
    ob, fb, _ = oracle.gla_fwd(q, k, v[..., 2:], la)
    assert _close(np.concatenate([oa, ob], -1), out)
    assert _close(np.concatenate([fa, fb], -1), fs)


def test_empty_sequence_returns_initial_state():
    q = np.zeros((2, 0, 3))
    v = np.zeros((2, 0, 2))
    s0 = _rng(14).standard_normal((2, 3, 2))
    out, fs, _ = oracle.gla_fwd(q, q, v, q, init_state=s0)
    assert out.shape == (2, 0, 2)
    assert _close(fs, s0)


# ---------------------------------------------------------------- golden worked examples

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["scalar_halving.json", "per_channel_2x2.json",
                                  "normalised_elu1.json"])
def test_golden_prefill(name):
    g = _golden(name)
    q = np.array(g["q"], float)[None]
    k = np.array(g["k"], float)[None]
    v = np.array(g["v"], float)[None]
    la = None if g["alpha"] is None else np.log(np.array(g["alpha"], float))[None]
    out, fs, fz = oracle.gla_fwd(q, k, v, la, feature_elu1=g.get("feature_elu1", False),
                                 normalize=g.get("normalize", False))
    assert _close(out[0], g["expect_out"], 1e-13)
    assert _close(fs[0], g["expect_final_state"], 1e-13)
    if "expect_final_z" in g:
        assert _close(fz[0], g["expect_final_z"], 1e-13)


def test_golden_decode():
    g = _golden("decode_step_2x2.json")
    o, st = oracle.gla_decode_step(np.array(g["q"], float), np.array(g["k"], float),
                                   np.array(g["v"], float), np.log(np.array(g["alpha"], float)),
                                   np.array(g["state"], float))
    assert _close(o, g["expect_out"], 1e-13)
    assert _close(st, g["expect_state"], 1e-13)
