"""GPU parity of the recurrent backward kernel (gla_bwd with GLA_FLAG_FORCE_SIMT,
and every call the chunk-form kernels do not take) against the fp64 oracle.

The kernel runs the recurrence token by token in fp32 on the same rounded
inputs the oracle receives.  dq, dk, dv and dinit are held to the fp32 bar
(relative L2 1e-5).  The gate gradient is a running sum over the remaining
tokens of q * dq - k * dk (fp32, up to L terms of either sign), held to
relative L2 1e-4."""
import numpy as np
import pytest

import causal_gated_linear_gb300 as gla
import oracle
import synth
from gpu_util import F32_REL, rel_l2, to_dev

pytestmark = pytest.mark.gpu

GATE_REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gla.load()


def _w(B, H, L, dk, dv, gate=True, init=True, dtype="bf16", seed=0):
    return synth.with_shape(synth.BWD, B=B, H=H, L=L, dk=dk, dv=dv, gate=gate, dtype=dtype,
                            init_std=0.1 if init else 0.0, seed=synth.BWD.seed + seed)


def run_bwd(w, x, want_dla=True, want_dinit=True, force_simt=True):
    import torch
    B, H, L, dk, dv = w.B, w.H, w.L, w.dk, w.dv
    q, k, v, do = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(x["dout"])
    la, s0, df = to_dev(x["log_alpha"]), to_dev(x["init_state"]), to_dev(x["dfinal"])
    nan = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device="cuda:0")
    dq, dk_, dv_ = nan(B, H, L, dk), nan(B, H, L, dk), nan(B, H, L, dv)
    dla = nan(B, H, L, dk) if (want_dla and la is not None) else None
    di = nan(B, H, dk, dv) if want_dinit else None
    if dla is not None and w.scalar_gate:
        dla = nan(B, H, L)
    gla.check(gla.gla_bwd(q, k, v, do, dq, dk_, dv_, B, H, L, dk, dv, log_alpha=la, init_state=s0, dfinal=df,
                          dlog_alpha=dla, dinit=di, in_dtype=gla.F32 if w.dtype == "f32" else gla.BF16,
                          flags=(gla.FLAG_SCALAR_GATE if w.scalar_gate else 0) |
                          (gla.FLAG_FORCE_SIMT if force_simt else 0)))
    torch.cuda.synchronize()
    gla.check(gla.gla_device_error())
    c = lambda t: None if t is None else t.cpu().numpy().astype(np.float64)
    return c(dq), c(dk_), c(dv_), c(dla), c(di)


def oracle_bwd(x):
    f = synth.as_f64
    return oracle.gla_bwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["dout"]), f(x["log_alpha"]),
                          f(x["init_state"]), f(x["dfinal"]))


def _check(got, ref, gate):
    for name, g, r in zip(("dq", "dk", "dv", "dlog_alpha", "dinit"), got, ref):
        if r is None or g is None:
            continue
        tol = GATE_REL if name == "dlog_alpha" else F32_REL
        assert rel_l2(g, r) <= tol, f"{name}: rel-L2 {rel_l2(g, r):.3e}"


@pytest.mark.parametrize("B,H,L,dk,dv,gate,init,dfin,dtype", [
    (1, 2, 1, 128, 128, True, True, True, "bf16"),
    (2, 1, 37, 64, 64, True, False, False, "bf16"),
    (1, 2, 100, 32, 32, False, True, True, "f32"),
    (1, 1, 257, 128, 64, True, True, True, "f32"),
    (2, 2, 16, 64, 128, True, True, False, "bf16"),
    (1, 1, 300, 32, 128, True, True, True, "bf16"),
    (1, 1, 129, 128, 32, True, False, True, "bf16"),
])
def test_bwd_shapes(B, H, L, dk, dv, gate, init, dfin, dtype):
    w = _w(B, H, L, dk, dv, gate, init, dtype, seed=L + dk + 3 * dv)
    x = synth.make_bwd(w, dfinal_std=0.5 if dfin else 0.0)
    _check(run_bwd(w, x), oracle_bwd(x), gate)


@pytest.mark.parametrize("B,H,L,dk,dv", [(1, 2, 77, 128, 128), (2, 1, 200, 64, 32), (1, 1, 16, 32, 64)])
def test_bwd_per_token_gate(B, H, L, dk, dv):
    """One gate per token (GLA_FLAG_SCALAR_GATE): the oracle runs on the gate
    broadcast to every channel, and the per-token gradient is the sum of its
    per-channel gradients."""
    w = synth.with_shape(_w(B, H, L, dk, dv, seed=L + 5), scalar_gate=True)
    x = synth.make_bwd(w, dfinal_std=0.5)
    got = run_bwd(w, x)
    xo = dict(x, log_alpha=np.repeat(x["log_alpha"][..., None], dk, axis=-1))
    ref = list(oracle_bwd(xo))
    ref[3] = ref[3].sum(axis=-1)
    _check(got, ref, True)


def test_bwd_optional_outputs_absent():
    """dlog_alpha and dinit NULL: the other gradients are unchanged."""
    w = _w(1, 2, 70, 64, 64, seed=11)
    x = synth.make_bwd(w, dfinal_std=0.5)
    full = run_bwd(w, x)
    part = run_bwd(w, x, want_dla=False, want_dinit=False)
    for a, b in zip(full[:3], part[:3]):
        assert np.array_equal(a, b)
    assert part[3] is None and part[4] is None


def test_bwd_empty_sequence():
    import torch
    df = torch.randn(2, 3, 64, 32, device="cuda:0")
    di = torch.full_like(df, float("nan"))
    gla.check(gla.gla_bwd(None, None, None, None, None, None, None, 2, 3, 0, 64, 32, dfinal=df, dinit=di))
    torch.cuda.synchronize()
    assert torch.equal(di, df)
    gla.check(gla.gla_bwd(None, None, None, None, None, None, None, 2, 3, 0, 64, 32, dinit=di))
    torch.cuda.synchronize()
    assert torch.count_nonzero(di).item() == 0


def test_bwd_rejects_bad_calls():
    import torch
    t = lambda *s: torch.zeros(s, dtype=torch.float32, device="cuda:0")
    q, k, v, do = t(1, 1, 8, 64), t(1, 1, 8, 64), t(1, 1, 8, 64), t(1, 1, 8, 64)
    dq, dk, dv = t(1, 1, 8, 64), t(1, 1, 8, 64), t(1, 1, 8, 64)
    F = gla.F32
    assert gla.gla_bwd(q, k, v, do, dq, dk, dv, 1, 1, 8, 48, 64, in_dtype=F) == gla.GLA_ERR_UNSUPPORTED
    assert gla.gla_bwd(q, k, v, do, dq, dk, None, 1, 1, 8, 64, 64, in_dtype=F) == gla.GLA_ERR_INVALID
    assert gla.gla_bwd(q, k, v, do, dq, dk, dv, 1, 1, 8, 64, 64, dlog_alpha=t(1, 1, 8, 64),
                       in_dtype=F) == gla.GLA_ERR_INVALID  # a gate gradient without a gate
    assert gla.gla_bwd(q, k, v, do, dq, dq, dv, 1, 1, 8, 64, 64, in_dtype=F) == gla.GLA_ERR_INVALID
    assert gla.gla_bwd(q, k, v, do, q, dk, dv, 1, 1, 8, 64, 64, in_dtype=F) == gla.GLA_ERR_INVALID
    assert gla.gla_bwd(q, k, v, do, dq.data_ptr() + 4, dk, dv, 1, 1, 8, 64, 64,
                       in_dtype=F) == gla.GLA_ERR_MISALIGNED
    assert gla.gla_bwd(q, k, v, do, dq, dk, dv, 1, 1, 8, 64, 64, in_dtype=F,
                       flags=gla.FLAG_NORMALIZE) == gla.GLA_ERR_INVALID
    assert gla.gla_bwd(q, k, v, do, dq, dk, dv, 1, 1, 8, 64, 64, in_dtype=F,
                       flags=gla.FLAG_FORCE_SIMT) == gla.GLA_OK


def test_bwd_full_sampled_and_homogeneity():
    """The backward workload (B8 H16 L4096 dk = dv = 128, bf16, gated), every head:
    with no initial state and no final-state gradient the loss sum <dout, o> is
    linear in q, in k and in v separately, so <dq, q> = <dk, k> = <dv, v> per head
    (three reductions made by different CTAs and sweeps); sampled heads against the
    oracle element by element."""
    w = synth.BWD
    x = synth.make_bwd(w)
    dq, dk, dv, dla, _ = run_bwd(w, x, want_dinit=False)
    f = synth.as_f64
    BH = w.B * w.H
    iq = np.einsum("hld,hld->h", dq.reshape(BH, w.L, w.dk), f(x["q"]).reshape(BH, w.L, w.dk))
    ik = np.einsum("hld,hld->h", dk.reshape(BH, w.L, w.dk), f(x["k"]).reshape(BH, w.L, w.dk))
    iv = np.einsum("hlj,hlj->h", dv.reshape(BH, w.L, w.dv), f(x["v"]).reshape(BH, w.L, w.dv))
    scale = np.abs(iq).max()
    assert np.max(np.abs(iq - iv)) <= 1e-5 * scale, np.max(np.abs(iq - iv)) / scale
    assert np.max(np.abs(ik - iv)) <= 1e-5 * scale, np.max(np.abs(ik - iv)) / scale
    heads = [0, 93]
    xs = synth.make_bwd(w, heads=heads)
    ref = oracle.gla_bwd(f(xs["q"]), f(xs["k"]), f(xs["v"]), f(xs["dout"]), f(xs["log_alpha"]))
    got = [None if a is None else a.reshape((BH,) + a.shape[2:])[heads] for a in (dq, dk, dv, dla)]
    _check(got + [None], list(ref[:4]) + [None], True)


@pytest.mark.parametrize("scalar", [False, True])
def test_bwd_deterministic_bitwise(scalar):
    """Two runs on the same inputs give bit-identical gradients.  With one gate per channel every
    output is a fixed-order fp32 computation; with one gate per token the token gradient is summed
    across the row blocks of a head by fp32 atomics (include/gla.h), so that one output is only
    held to the fp32 bar between runs and every other output must still be bit-identical."""
    w = synth.with_shape(_w(1, 3, 333, 128, 128, seed=41), scalar_gate=scalar)
    x = synth.make_bwd(w, dfinal_std=0.5)
    a = run_bwd(w, x)
    b = run_bwd(w, x)
    for name, ga, gb in zip(("dq", "dk", "dv", "dlog_alpha", "dinit"), a, b):
        if scalar and name == "dlog_alpha":
            assert rel_l2(ga, gb) <= F32_REL, name
        else:
            assert np.array_equal(ga, gb), name
