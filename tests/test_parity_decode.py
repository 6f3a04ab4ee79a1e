"""GPU parity of the decode step (gla_decode_step) against the fp64 oracle."""
import numpy as np
import pytest

import causal_gated_linear_gb300 as gla
import oracle
import synth
from gpu_util import F32_REL, assert_bf16_close, rel_l2, run_prefill, to_dev

pytestmark = pytest.mark.gpu

DEC_REL = 1e-5  # fp32 state and output: the step is plain fp32 FMA


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gla.load()


@pytest.mark.parametrize("NS,H,dk,dv", [(3, 2, 128, 128), (2, 3, 64, 32), (1, 2, 100, 12),
                                        (2, 1, 256, 512)])
def test_decode_shapes(NS, H, dk, dv):
    import torch
    st0 = synth.decode_state(NS, H, dk, dv, 0.1, seed=3)
    st = to_dev(st0)
    ref = st0.astype(np.float64)
    for step in range(4):
        tok = synth.decode_token(NS, H, dk, dv, step, seed=3)
        out = torch.full((NS, H, dv), float("nan"), device="cuda:0")
        gla.check(gla.gla_decode_step(to_dev(tok["q"]), to_dev(tok["k"]), to_dev(tok["v"]),
                                      to_dev(tok["log_alpha"]), st, out, NS, H, dk, dv))
        torch.cuda.synchronize()
        ro, ref = oracle.gla_decode_step(synth.as_f64(tok["q"]), synth.as_f64(tok["k"]),
                                         synth.as_f64(tok["v"]), synth.as_f64(tok["log_alpha"]), ref)
        assert rel_l2(out.cpu().numpy(), ro) <= DEC_REL
    assert rel_l2(st.cpu().numpy(), ref) <= DEC_REL


def test_decode_no_gate():
    import torch
    st0 = synth.decode_state(2, 2, 64, 64, 0.1, seed=4)
    st = to_dev(st0)
    tok = synth.decode_token(2, 2, 64, 64, 0, seed=4)
    out = torch.empty((2, 2, 64), device="cuda:0")
    gla.check(gla.gla_decode_step(to_dev(tok["q"]), to_dev(tok["k"]), to_dev(tok["v"]), None, st, out,
                                  2, 2, 64, 64))
    torch.cuda.synchronize()
    ro, rs = oracle.gla_decode_step(synth.as_f64(tok["q"]), synth.as_f64(tok["k"]),
                                    synth.as_f64(tok["v"]), None, st0)
    assert rel_l2(out.cpu().numpy(), ro) <= DEC_REL and rel_l2(st.cpu().numpy(), rs) <= DEC_REL


def test_decode_full_1024_steps_sampled():
    """Full decode workload: 256 x 32 heads, 1024 steps; every step's output is
    checked on a sample of heads, and the final state on the same sample."""
    import torch
    d = synth.DECODE
    NS, H, dk, dv, seed = d["NS"], d["H"], d["dk"], d["dv"], d["seed"]
    st = to_dev(synth.decode_state(NS, H, dk, dv, d["state_std"], seed))
    heads = [0, 1, 777, 4095, 5000, 8191]
    ref = synth.decode_state(NS, H, dk, dv, d["state_std"], seed, heads=heads).astype(np.float64)
    out = torch.empty((NS, H, dv), device="cuda:0")
    sel = torch.tensor(heads, device="cuda:0")
    worst = 0.0
    for step in range(d["steps"]):
        tok = synth.decode_token(NS, H, dk, dv, step, seed, d["gate_mean"], d["gate_std"])
        gla.check(gla.gla_decode_step(to_dev(tok["q"]), to_dev(tok["k"]), to_dev(tok["v"]),
                                      to_dev(tok["log_alpha"]), st, out, NS, H, dk, dv))
        got = out.view(NS * H, dv).index_select(0, sel).cpu().numpy()
        ts = synth.decode_token(NS, H, dk, dv, step, seed, d["gate_mean"], d["gate_std"], heads=heads)
        ro, ref = oracle.gla_decode_step(synth.as_f64(ts["q"]), synth.as_f64(ts["k"]),
                                         synth.as_f64(ts["v"]), synth.as_f64(ts["log_alpha"]), ref)
        worst = max(worst, rel_l2(got, ro))
    assert worst <= DEC_REL, worst
    s = st.view(NS * H, dk, dv).index_select(0, sel).cpu().numpy()
    assert rel_l2(s, ref) <= DEC_REL


def test_decode_steps_equal_prefill():
    """N decode steps from an initial state reproduce the prefill of the same N tokens."""
    import torch
    w = synth.with_shape(synth.PREFILL, B=1, H=2, L=40, init_std=0.1, seed=81)
    x = synth.make_prefill(w)
    o, s, _ = run_prefill(w, x, out_f32=True)
    st = to_dev(x["init_state"]).clone()
    outs = []
    for t in range(40):
        out = torch.empty((1, 2, 128), device="cuda:0")
        gla.check(gla.gla_decode_step(to_dev(np.ascontiguousarray(x["q"][:, :, t])),
                                      to_dev(np.ascontiguousarray(x["k"][:, :, t])),
                                      to_dev(np.ascontiguousarray(x["v"][:, :, t])),
                                      to_dev(np.ascontiguousarray(x["log_alpha"][:, :, t])), st, out,
                                      1, 2, 128, 128))
        outs.append(out.cpu().numpy())
    dec = np.stack(outs, axis=2)
    assert_bf16_close(dec, o, "decode vs prefill out")
    assert_bf16_close(st.cpu().numpy(), s, "decode vs prefill state")
