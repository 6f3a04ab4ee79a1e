"""Planted mistakes: each deliberately wrong oracle variant must fail a pin.

The variants are compiled from the oracle source with -DORACLE_PLANT=n into a
temporary directory (CPU only).  This shows the pins in test_oracle_pins.py
are sharp enough to catch a dropped term, a wrong index or an off-by-one in
the decay range.
"""
import json
import os

import numpy as np
import pytest

import oracle
from test_oracle_pins import _close, _golden, _inputs, _phi, quadratic_masked


@pytest.fixture(scope="module")
def plant_dir(tmp_path_factory):
    d = str(tmp_path_factory.mktemp("plants"))
    for n in (1, 2, 3, 4, 5, 6, 7, 8):
        oracle.build(plant=n, build_dir=d)
    return d


def _fwd(plant, d, *a, **kw):
    return oracle.gla_fwd(*a, plant=plant, build_dir=d, **kw)


def test_plant1_decay_after_write_is_caught(plant_dir):
    q, k, v, la = _inputs(2, 64, 6, 4)
    out, _, _ = _fwd(1, plant_dir, q, k, v, la)
    assert not _close(out, quadratic_masked(q, k, v, la))
    g = _golden("scalar_halving.json")
    o, _, _ = _fwd(1, plant_dir, np.array(g["q"], float)[None], np.array(g["k"], float)[None],
                   np.array(g["v"], float)[None], np.log(np.array(g["alpha"], float))[None])
    assert not _close(o[0], g["expect_out"], 1e-13)


def test_plant2_transposed_contraction_is_caught(plant_dir):
    g = _golden("per_channel_2x2.json")
    o, _, _ = _fwd(2, plant_dir, np.array(g["q"], float)[None], np.array(g["k"], float)[None],
                   np.array(g["v"], float)[None], np.log(np.array(g["alpha"], float))[None])
    assert not _close(o[0], g["expect_out"], 1e-13)
    q, k, v, _ = _inputs(4, 29, 6, 6, gate=False)
    out, _, _ = _fwd(2, plant_dir, q, k, v)
    S = np.cumsum(np.einsum("bld,blj->bldj", k, v), axis=1)
    assert not _close(out, np.einsum("bld,bldj->blj", q, S))


def test_plant3_dropped_normaliser_is_caught(plant_dir):
    q, k, v, _ = _inputs(5, 50, 4, 3, gate=False)
    out, _, _ = _fwd(3, plant_dir, q, k, v, feature_elu1=True, normalize=True)
    pq, pk = _phi(q), _phi(k)
    sim = np.tril(pq[0] @ pk[0].T)
    assert not _close(out[0], (sim @ v[0]) / sim.sum(axis=1, keepdims=True))


def test_plant4_exclusive_output_is_caught(plant_dir):
    q, k, v, _ = _inputs(1, 37, 5, 3, gate=False)
    out, _, _ = _fwd(4, plant_dir, q, k, v)
    S = np.cumsum(np.einsum("bld,blj->bldj", k, v), axis=1)
    assert not _close(out, np.einsum("bld,bldj->blj", q, S))


def test_plant5_delta_prediction_dropped_is_caught(plant_dir):
    from test_oracle_delta_pins import _close as dclose, _inputs as dinputs, triangular_form
    q, k, v, beta = dinputs(1, 40, 6, 5)
    out, fs = oracle.delta_fwd(q, k, v, beta, plant=5, build_dir=plant_dir)
    O, S = triangular_form(q[0], k[0], v[0], beta[0], np.zeros((6, 5)))
    assert not dclose(out[0], O)
    g = _golden("delta_2x2.json")
    o, _ = oracle.delta_fwd(*(np.array(g[n], float)[None] for n in ("q", "k", "v", "beta")),
                            plant=5, build_dir=plant_dir)
    assert not dclose(o[0], g["expect_out"], 1e-14)


def test_plant6_delta_output_before_write_is_caught(plant_dir):
    from test_oracle_delta_pins import _close as dclose
    g = _golden("delta_2x2.json")
    o, _ = oracle.delta_fwd(*(np.array(g[n], float)[None] for n in ("q", "k", "v", "beta")),
                            plant=6, build_dir=plant_dir)
    assert not dclose(o[0], g["expect_out"], 1e-14)


def _bwd_vs_fd(plant, d):
    from test_oracle_bwd_pins import _fd, _inputs as binputs, _loss
    q, k, v, la, s0, Wo, Wf = binputs(5, L=6, dk=3, dv=2)
    got = oracle.gla_bwd(q, k, v, Wo, la, s0, Wf, plant=plant, build_dir=d)
    f = lambda: _loss(q, k, v, la, s0, Wo, Wf)
    refs = (_fd(f, q), _fd(f, k), _fd(f, v), _fd(f, la), _fd(f, s0))
    return [float(np.max(np.abs(g - r))) for g, r in zip(got, refs)]


def test_plant7_gate_gradient_with_wrong_state_is_caught(plant_dir):
    err = _bwd_vs_fd(7, plant_dir)
    assert err[3] > 1e-3, err


def test_plant8_undecayed_state_gradient_is_caught(plant_dir):
    err = _bwd_vs_fd(8, plant_dir)
    assert max(err[1], err[2], err[4]) > 1e-3, err
