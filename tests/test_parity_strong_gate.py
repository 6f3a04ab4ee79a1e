"""GPU parity of the chunk kernels for gates that decay strongly inside one chunk.

"Gated Linear Attention", GLA Recurrent Form: alpha_t lies in (0, 1) with no
lower bound, so a channel can lose almost all of its state within one chunk
(e^{b_C} below e^-64 over 64 tokens).  The tensor-core prefill then takes that
channel's factors relative to the chunk start and adds its intra-chunk scores
with exponents <= 0; these tests hold it to the bf16 bar against the fp64
oracle on such gates, on both value-tile widths, with one gate per channel and
with one gate per token.

Cases: log alpha = -1e4 on every channel (every token forgets everything before
it, so o_t = (q_t . k_t) v_t: also checked against that closed form); a
constant alpha = 0.1 (b_C = 64 ln 0.1 = -147 per chunk); strong decay on a
subset of the channels only; strong decay in some chunks only.
"""
import numpy as np
import pytest

import causal_gated_linear_gb300 as gla
import synth
from gpu_util import assert_bf16_close, oracle_prefill, rel_l2, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gla.load()


def _inputs(L, dk, dv, H=2, init=True, scalar=False, seed=0, elu=False):
    w = synth.with_shape(synth.PREFILL, B=1, H=H, L=L, dk=dk, dv=dv, init_std=0.1 if init else 0.0,
                         scalar_gate=scalar, feature_elu1=elu, normalize=elu, qk_scale=not elu,
                         seed=900 + seed + L + dk + dv)
    return w, synth.make_prefill(w)


def _with_gate(x, la):
    y = dict(x)
    y["log_alpha"] = np.ascontiguousarray(la, dtype=np.float32)
    return y


def _check(w, x, dvt, monkeypatch):
    monkeypatch.setenv("GLA_TC_DVT", dvt)
    o, s, _ = run_prefill(w, x, flags=gla.FLAG_FORCE_CHUNK)
    assert np.isfinite(o).all() and np.isfinite(s).all()
    ro, rs, _ = oracle_prefill(w, x)
    assert_bf16_close(o, ro, "out")
    if w.normalize:
        # phi >= 0 makes the unnormalised state grow with L (|S| ~ 40 here), so its bf16-operand
        # rounding is held to the relative bar only, as in the other normalised tests
        assert rel_l2(s, rs) <= 1e-2, rel_l2(s, rs)
    else:
        assert_bf16_close(s, rs, "state")
    return o, s


DVT = ["64", "128"]
SHAPES = [(200, 128, 128), (130, 64, 64), (64, 128, 256)]


@pytest.mark.parametrize("dvt", DVT)
@pytest.mark.parametrize("L,dk,dv", SHAPES)
def test_forget_everything(monkeypatch, dvt, L, dk, dv):
    """log alpha = -1e4: o_t = (q_t . k_t) v_t and the final state is k_{L-1} v_{L-1}^T."""
    w, x = _inputs(L, dk, dv)
    x = _with_gate(x, np.full(x["log_alpha"].shape, -1e4))
    o, s = _check(w, x, dvt, monkeypatch)
    q, k, v = (synth.as_f64(x[n]).reshape(2, L, -1) for n in ("q", "k", "v"))
    closed = np.einsum("hld,hld->hl", q, k)[..., None] * v
    assert_bf16_close(o.reshape(2, L, dv), closed, "closed form")
    assert_bf16_close(s.reshape(2, dk, dv), np.einsum("hd,hj->hdj", k[:, -1], v[:, -1]), "closed-form state")


@pytest.mark.parametrize("dvt", DVT)
@pytest.mark.parametrize("L,dk,dv", SHAPES)
def test_constant_alpha_0p1(monkeypatch, dvt, L, dk, dv):
    """alpha = 0.1 on every channel: each chunk decays by e^-147."""
    w, x = _inputs(L, dk, dv, seed=1)
    _check(w, _with_gate(x, np.full(x["log_alpha"].shape, np.log(0.1))), dvt, monkeypatch)


@pytest.mark.parametrize("dvt", DVT)
@pytest.mark.parametrize("strong", [-1e4, -3.0, -1.2])
def test_some_channels_strong(monkeypatch, dvt, strong):
    """The workload's gate on most channels, a strong constant gate on every third one and
    on the last quad (mixes strong and ordinary channels in one thread's four)."""
    L, dk, dv = 200, 128, 128
    w, x = _inputs(L, dk, dv, seed=2)
    la = x["log_alpha"].copy()
    la[..., ::3] = strong
    la[..., -4:-1] = strong
    _check(w, _with_gate(x, la), dvt, monkeypatch)


@pytest.mark.parametrize("dvt", DVT)
def test_some_chunks_strong(monkeypatch, dvt):
    """Strong decay only in tokens [70, 170) (all channels) and [256, 260) (channel 5): chunks 1,
    2 and 4 take the strong path, chunks 0 and 3 the ordinary one; the state carries across
    both kinds."""
    L, dk, dv = 300, 128, 128
    w, x = _inputs(L, dk, dv, seed=3)
    la = x["log_alpha"].copy()
    la[:, :, 70:170, :] = -2.0
    la[:, :, 256:260, 5] = -1e4
    _check(w, _with_gate(x, la), dvt, monkeypatch)


@pytest.mark.parametrize("dvt", DVT)
@pytest.mark.parametrize("gate", [-1e4, np.log(0.1), "mixed"])
def test_per_token_gate_strong(monkeypatch, dvt, gate):
    """One gate per token (GLA_FLAG_SCALAR_GATE) with strong decay."""
    L, dk, dv = 200, 128, 128
    w, x = _inputs(L, dk, dv, scalar=True, seed=4)
    la = x["log_alpha"].copy()
    if gate == "mixed":
        la[:, :, 64:128] = -5.0
    else:
        la[...] = gate
    _check(w, _with_gate(x, la), dvt, monkeypatch)


def test_feature_map_with_strong_gate(monkeypatch):
    """phi = elu + 1 and the normaliser with a strong gate on every other channel (the strong
    scores apply phi to the raw inputs; z decays with the state)."""
    L, dk, dv = 150, 64, 64
    w, x = _inputs(L, dk, dv, seed=5, elu=True)
    la = x["log_alpha"].copy()
    la[..., 1::2] = -4.0
    _check(w, _with_gate(x, la), "64", monkeypatch)


def test_long_strong_sequence(monkeypatch):
    """A longer sequence (32 chunks) at alpha = 0.1: the strong path keeps up with the pipeline."""
    L, dk, dv = 2048, 128, 128
    w, x = _inputs(L, dk, dv, H=1, seed=6)
    _check(w, _with_gate(x, np.full(x["log_alpha"].shape, np.log(0.1))), "64", monkeypatch)
