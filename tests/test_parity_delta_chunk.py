"""GPU parity of the delta rule in chunk form on the tensor cores (gla_delta_fwd
with d_k = d_v = 128) against the fp64 oracle.

"linear-attention" blog, Delta attention and its Prefill section: the writes of
a chunk solve one unit lower-triangular system; the kernel inverts it per chunk
(fp32) and runs every product on bf16 tensor cores with fp32 accumulation and an
fp32 state, so outputs and final states are held to the bf16 bar (relative L2
<= 1e-2, max-abs <= 5e-2).  Gates that decay by more than e^-64 within a chunk
send their head to the token-by-token kernel.
"""
import numpy as np
import pytest

import causal_gated_linear_gb300 as gla
import oracle
import synth
from gpu_util import assert_bf16_close, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gla.load()


def _w(B, H, L, gate=True, init=True, seed=0):
    return synth.with_shape(synth.DELTA, B=B, H=H, L=L, gate=gate, init_std=0.1 if init else 0.0,
                            seed=synth.DELTA.seed + 700 + seed)


def run(w, x, out_f32=False, force_simt=False, in_place=False):
    import torch
    q, k, v, b = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(x["beta"])
    la, s0 = to_dev(x["log_alpha"]), to_dev(x["init_state"])
    odt = torch.float32 if out_f32 else torch.bfloat16
    out = torch.full((w.B, w.H, w.L, w.dv), float("nan"), dtype=odt, device="cuda:0")
    fs = s0 if in_place else torch.full((w.B, w.H, w.dk, w.dv), float("nan"), dtype=torch.float32, device="cuda:0")
    gla.check(gla.gla_delta_fwd(q, k, v, b, out, w.B, w.H, w.L, w.dk, w.dv, log_alpha=la, init_state=s0,
                                final_state=fs, out_dtype=gla.F32 if out_f32 else gla.BF16,
                                flags=gla.FLAG_FORCE_SIMT if force_simt else 0))
    torch.cuda.synchronize()
    gla.check(gla.gla_device_error())
    return out.float().cpu().numpy().astype(np.float64), fs.cpu().numpy().astype(np.float64)


def ref(x):
    f = synth.as_f64
    return oracle.delta_fwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["beta"]), f(x["log_alpha"]), f(x["init_state"]))


@pytest.mark.parametrize("B,H,L,gate,init,out_f32", [
    (1, 2, 64, True, True, False),
    (1, 2, 200, True, False, True),
    (2, 1, 65, True, True, False),
    (1, 1, 1, True, True, True),
    (1, 3, 513, False, True, False),
    (1, 1, 130, False, False, True),
])
def test_delta_chunk_shapes(B, H, L, gate, init, out_f32):
    w = _w(B, H, L, gate, init, seed=L)
    x = synth.make_delta(w)
    o, s = run(w, x, out_f32=out_f32)
    ro, rs = ref(x)
    assert_bf16_close(o, ro, "out")
    assert_bf16_close(s, rs, "state")


def test_delta_chunk_matches_token_kernel_and_in_place_state():
    w = _w(1, 2, 300, seed=7)
    x = synth.make_delta(w)
    o1, s1 = run(w, x)
    o2, s2 = run(w, x, force_simt=True)
    assert_bf16_close(o1, o2, "out vs token-by-token")
    assert_bf16_close(s1, s2, "state vs token-by-token")
    o3, s3 = run(w, x, in_place=True)
    assert np.array_equal(o3, o1) and np.array_equal(s3, s1)


@pytest.mark.parametrize("gate", [-1e4, float(np.log(0.1)), "one head"])
def test_delta_chunk_strong_gates_exact(gate):
    w = _w(1, 3, 200, seed=9)
    x = synth.make_delta(w)
    la = x["log_alpha"].copy()
    if gate == "one head":
        la[0, 1, 64:128, ::3] = -3.0
    else:
        la[...] = gate
    x["log_alpha"] = la.astype(np.float32)
    o, s = run(w, x, out_f32=True)
    ro, rs = ref(x)
    assert_bf16_close(o, ro, "out")
    assert_bf16_close(s, rs, "state")


def test_delta_chunk_beta_zero_only_decays():
    """beta = 0: nothing is written (T = I, U = 0), the state only decays (closed form)."""
    w = _w(1, 2, 150, seed=5)
    x = synth.make_delta(w)
    x["beta"] = np.zeros_like(x["beta"])
    o, s = run(w, x, out_f32=True)
    la = synth.as_f64(x["log_alpha"])[0]
    dec = np.exp(np.cumsum(la, axis=1))
    s0 = synth.as_f64(x["init_state"])[0]
    q = synth.as_f64(x["q"])[0]
    assert_bf16_close(o[0], np.einsum("btd,btd,bdj->btj", q, dec, s0), "out")
    assert_bf16_close(s[0], dec[:, -1][..., None] * s0, "state")


def test_delta_chunk_deterministic_bitwise():
    w = _w(1, 3, 333, seed=10)
    x = synth.make_delta(w)
    a, b = run(w, x), run(w, x)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_delta_chunk_full_sampled():
    """The delta workload (B8 H16 L4096 d128, gated, unit keys), sampled heads."""
    w = synth.DELTA
    x = synth.make_delta(w)
    o, s = run(w, x, out_f32=True)
    heads = [0, 77, 127]
    xs = synth.make_delta(w, heads=heads)
    ro, rs = oracle.delta_fwd(synth.as_f64(xs["q"]), synth.as_f64(xs["k"]), synth.as_f64(xs["v"]),
                              synth.as_f64(xs["beta"]), synth.as_f64(xs["log_alpha"]), None)
    o = o.reshape(w.B * w.H, w.L, w.dv)[heads]
    s = s.reshape(w.B * w.H, w.dk, w.dv)[heads]
    assert_bf16_close(o, ro, "out")
    assert_bf16_close(s, rs, "state")
