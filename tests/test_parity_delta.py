"""GPU parity of the token-by-token delta-rule kernel (gla_delta_fwd_ex with
GLA_FLAG_FORCE_SIMT, and every shape the chunk form does not take) against the
fp64 oracle.

The kernel runs the recurrence token by token in fp32 on the same rounded
inputs the oracle receives, so fp32 output is held to relative L2 1e-5 on
sequences of a few hundred tokens; bf16 output to the bf16 bar."""
import numpy as np
import pytest

import causal_gated_linear_gb300 as gla
import oracle
import synth
from gpu_util import F32_REL, assert_bf16_close, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gla.load()


def _w(B, H, L, dk, dv, gate=True, init=True, seed=0):
    return synth.with_shape(synth.DELTA, B=B, H=H, L=L, dk=dk, dv=dv, gate=gate,
                            init_std=0.1 if init else 0.0, seed=synth.DELTA.seed + seed)


def run_delta(w, x, out_f32=False, in_place=False, force_simt=True):
    import torch
    q, k, v, b = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(x["beta"])
    la, s0 = to_dev(x["log_alpha"]), to_dev(x["init_state"])
    odt = torch.float32 if out_f32 else torch.bfloat16
    out = torch.full((w.B, w.H, w.L, w.dv), float("nan"), dtype=odt, device="cuda:0")
    if in_place:
        fs = s0
    else:
        fs = torch.full((w.B, w.H, w.dk, w.dv), float("nan"), dtype=torch.float32, device="cuda:0")
    gla.check(gla.gla_delta_fwd(q, k, v, b, out, w.B, w.H, w.L, w.dk, w.dv, log_alpha=la, init_state=s0,
                                final_state=fs, out_dtype=gla.F32 if out_f32 else gla.BF16,
                                flags=gla.FLAG_FORCE_SIMT if force_simt else 0))
    torch.cuda.synchronize()
    gla.check(gla.gla_device_error())
    return out.float().cpu().numpy().astype(np.float64), fs.cpu().numpy().astype(np.float64)


def oracle_delta(w, x):
    return oracle.delta_fwd(synth.as_f64(x["q"]), synth.as_f64(x["k"]), synth.as_f64(x["v"]),
                            synth.as_f64(x["beta"]), synth.as_f64(x["log_alpha"]), synth.as_f64(x["init_state"]))


@pytest.mark.parametrize("B,H,L,dk,dv,gate,init", [
    (2, 3, 1, 128, 128, True, True),
    (1, 2, 31, 128, 128, True, False),
    (1, 2, 33, 64, 64, False, True),
    (2, 1, 100, 32, 16, True, True),
    (1, 2, 257, 128, 80, True, True),
    (1, 1, 130, 64, 192, True, False),
])
def test_delta_shapes_fp32_out(B, H, L, dk, dv, gate, init):
    w = _w(B, H, L, dk, dv, gate, init, seed=L + dk + dv)
    x = synth.make_delta(w)
    o, s = run_delta(w, x, out_f32=True)
    ro, rs = oracle_delta(w, x)
    assert rel_l2(o, ro) <= F32_REL, rel_l2(o, ro)
    assert rel_l2(s, rs) <= F32_REL, rel_l2(s, rs)


def test_delta_bf16_out_and_in_place_state():
    w = _w(2, 2, 77, 128, 128, seed=3)
    x = synth.make_delta(w)
    ro, rs = oracle_delta(w, x)
    o, s = run_delta(w, x, in_place=True)
    assert_bf16_close(o, ro, "out")
    assert rel_l2(s, rs) <= F32_REL


def test_delta_empty_sequence_copies_state():
    import torch
    s0 = torch.randn(2, 2, 64, 64, device="cuda:0")
    fs = torch.full_like(s0, float("nan"))
    gla.check(gla.gla_delta_fwd(None, None, None, None, None, 2, 2, 0, 64, 64, init_state=s0, final_state=fs))
    torch.cuda.synchronize()
    assert torch.equal(fs, s0)


def test_delta_beta_zero_only_decays():
    """beta = 0 on the GPU: nothing is written, the state only decays (closed form)."""
    w = _w(1, 2, 40, 64, 64, seed=5)
    x = synth.make_delta(w)
    x["beta"] = np.zeros_like(x["beta"])
    o, s = run_delta(w, x, out_f32=True)
    la = synth.as_f64(x["log_alpha"])[0]
    dec = np.exp(np.cumsum(la, axis=1))
    s0 = synth.as_f64(x["init_state"])[0]
    q = synth.as_f64(x["q"])[0]
    assert rel_l2(o[0], np.einsum("btd,btd,bdj->btj", q, dec, s0)) <= F32_REL
    assert rel_l2(s[0], dec[:, -1][..., None] * s0) <= F32_REL


def test_delta_full_sampled():
    """The delta workload (B8 H16 L4096 dk = dv = 128, gated, unit keys), sampled heads."""
    w = synth.DELTA
    x = synth.make_delta(w)
    o, s = run_delta(w, x, out_f32=True)
    heads = [0, 77, 127]
    xs = synth.make_delta(w, heads=heads)
    ro, rs = oracle.delta_fwd(synth.as_f64(xs["q"]), synth.as_f64(xs["k"]), synth.as_f64(xs["v"]),
                              synth.as_f64(xs["beta"]), synth.as_f64(xs["log_alpha"]), None)
    o = o.reshape(w.B * w.H, w.L, w.dv)[heads]
    s = s.reshape(w.B * w.H, w.dk, w.dv)[heads]
    assert rel_l2(o, ro) <= F32_REL, rel_l2(o, ro)
    assert rel_l2(s, rs) <= F32_REL, rel_l2(s, rs)
