"""gla_fwd_host: host buffers in, host buffers out, copies overlapped with the
computation over head groups.  Every head is an independent problem computed
by the same kernels, so the results equal gla_fwd_ex's on device buffers bit
for bit, whatever the grouping."""
import numpy as np
import pytest

import causal_gated_linear_gb300 as gla
import synth
from gpu_util import run_prefill, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gla.load()


def _host(x):
    import torch
    if x is None:
        return None
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


def run_host(w, x, groups, flags=0, init_z=None, final_z=False, streams=None):
    import torch
    B, H, L, dk, dv = w.B, w.H, w.L, w.dk, w.dv
    f32in = w.dtype == "f32"
    odt = torch.float32 if f32in else torch.bfloat16
    host = dict(q=_host(x["q"]), k=_host(x["k"]), v=_host(x["v"]), log_alpha=_host(x["log_alpha"]),
                init_state=_host(x["init_state"]), init_z=_host(init_z))
    host["out"] = torch.full((B, H, L, dv), float("nan"), dtype=odt).pin_memory()
    host["final_state"] = torch.full((B, H, dk, dv), float("nan")).pin_memory()
    if final_z:
        host["final_z"] = torch.full((B, H, dk), float("nan")).pin_memory()
    dev = {n: (None if t is None else torch.empty(t.shape, dtype=t.dtype, device="cuda:0"))
           for n, t in host.items()}
    fl = flags | (gla.FLAG_FEATURE_ELU1 if w.feature_elu1 else 0) | (gla.FLAG_NORMALIZE if w.normalize else 0) | \
        (gla.FLAG_SCALAR_GATE if w.scalar_gate else 0)
    s = streams or [torch.cuda.Stream() for _ in range(3)]
    st = gla.gla_fwd_host({n: t for n, t in host.items() if t is not None},
                          {n: t for n, t in dev.items() if t is not None}, B, H, L, dk, dv, chunk=w.chunk,
                          groups=groups, in_dtype=gla.F32 if f32in else gla.BF16,
                          out_dtype=gla.F32 if f32in else gla.BF16, flags=fl, copy_in=s[0], compute=s[1],
                          copy_out=s[2])
    return st, host, dev, s


def _np(t):
    return None if t is None else t.float().numpy().astype(np.float64)


@pytest.mark.parametrize("groups", [1, 3, 8, 1000])
def test_host_pipeline_equals_device_call(groups):
    import torch
    w = synth.with_shape(synth.PREFILL, B=2, H=3, L=200, init_std=0.1)
    x = synth.make_prefill(w)
    st, host, _, _ = run_host(w, x, groups)
    gla.check(st)
    torch.cuda.synchronize()
    gla.check(gla.gla_device_error())
    o, s, _ = run_prefill(w, x)
    assert np.array_equal(_np(host["out"]), o)
    assert np.array_equal(_np(host["final_state"]), s)


@pytest.mark.parametrize("case", ["scalar_gate", "elu_norm", "fp32", "short"])
def test_host_pipeline_variants(case):
    import torch
    z0 = None
    if case == "scalar_gate":
        w = synth.with_shape(synth.PREFILL, B=1, H=4, L=130, scalar_gate=True, init_std=0.1)
    elif case == "elu_norm":
        w = synth.with_shape(synth.ELU_NORM, B=2, H=2, L=100)
        z0 = np.abs(synth.to_f32(synth.normals(5, 9, (2 * 2 * 64,)))).reshape(2, 2, 64)
    elif case == "fp32":
        w = synth.with_shape(synth.FP32_SMALL, B=1, H=3, L=70, init_std=0.1)
    else:
        w = synth.with_shape(synth.PREFILL, B=2, H=4, L=8, init_std=0.1)
    x = synth.make_prefill(w)
    st, host, _, _ = run_host(w, x, 3, init_z=z0, final_z=w.normalize)
    gla.check(st)
    torch.cuda.synchronize()
    gla.check(gla.gla_device_error())
    o, s, fz = run_prefill(w, x, final_z=w.normalize, init_z=z0)
    assert np.array_equal(_np(host["out"]), o)
    assert np.array_equal(_np(host["final_state"]), s)
    if w.normalize:
        assert np.array_equal(_np(host["final_z"]), fz)


def test_host_pipeline_back_to_back_reuses_staging():
    """Two calls queued without a host synchronisation in between, on the same
    staging buffers and streams, with different inputs: each host output
    matches its own inputs."""
    import torch
    w = synth.with_shape(synth.PREFILL, B=1, H=6, L=300, init_std=0.1)
    xa = synth.make_prefill(w)
    xb = synth.make_prefill(synth.with_shape(w, seed=w.seed + 1))
    st, ha, dev, s = run_host(w, xa, 4)
    gla.check(st)
    hb = {n: (None if t is None else (_host(xb[n]) if n in xb else torch.full_like(t, float("nan")).pin_memory()))
          for n, t in ha.items()}
    fl = gla.FLAG_SCALAR_GATE if w.scalar_gate else 0
    gla.check(gla.gla_fwd_host({n: t for n, t in hb.items() if t is not None},
                               {n: t for n, t in dev.items() if t is not None}, w.B, w.H, w.L, w.dk, w.dv,
                               groups=4, flags=fl, copy_in=s[0], compute=s[1], copy_out=s[2]))
    torch.cuda.synchronize()
    gla.check(gla.gla_device_error())
    for h, x in ((ha, xa), (hb, xb)):
        o, fs, _ = run_prefill(w, x)
        assert np.array_equal(_np(h["out"]), o)
        assert np.array_equal(_np(h["final_state"]), fs)


def test_host_pipeline_rejects_bad_calls():
    import torch
    w = synth.with_shape(synth.PREFILL, B=1, H=2, L=64, init_std=0.1)
    x = synth.make_prefill(w)
    host = dict(q=_host(x["q"]), k=_host(x["k"]), v=_host(x["v"]), log_alpha=_host(x["log_alpha"]),
                init_state=_host(x["init_state"]),
                out=torch.empty(1, 2, 64, 128, dtype=torch.bfloat16).pin_memory(),
                final_state=torch.empty(1, 2, 128, 128).pin_memory())
    dev = {n: torch.empty(t.shape, dtype=t.dtype, device="cuda:0") for n, t in host.items()}
    args = (1, 2, 64, 128, 128)
    assert gla.gla_fwd_host(host, dev, *args, groups=0) == gla.GLA_ERR_INVALID
    assert gla.gla_fwd_host(host, {n: t for n, t in dev.items() if n != "init_state"}, *args) == \
        gla.GLA_ERR_INVALID  # a buffer on one side only
    alias = dict(dev, final_state=dev["init_state"])
    assert gla.gla_fwd_host(host, alias, *args) == gla.GLA_ERR_INVALID
    ha = {n: t for n, t in host.items()}
    assert gla.load().gla_fwd_host(None, None, 1, None, None, None) == gla.GLA_ERR_INVALID
    assert gla.gla_fwd_host(ha, dev, 1, 2, 64, 128, 128, chunk=32) == gla.GLA_ERR_UNSUPPORTED
