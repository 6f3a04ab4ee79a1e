"""Helpers shared by the GPU parity tests: upload generated inputs, run the
C-ABI entry points, and compare with the oracle by relative L2 / max-abs."""
from __future__ import annotations

import numpy as np

import causal_gated_linear_gb300 as gla
import oracle
import synth

# tolerances of the bf16 path (relative L2 and max-abs) and the fp32 path
BF16_REL, BF16_ABS = 1e-2, 5e-2
F32_REL = 1e-5


def dev():
    import torch
    return torch.device("cuda:0")


def to_dev(x):
    import torch
    if x is None:
        return None
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev())
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev())


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (n if n > 0 else 1.0))


def max_abs(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(x - ref))) if x.size else 0.0


def assert_bf16_close(x, ref, what=""):
    r, a = rel_l2(x, ref), max_abs(x, ref)
    assert r <= BF16_REL and a <= BF16_ABS, f"{what}: rel-L2 {r:.3e} max-abs {a:.3e}"
    return r, a


def run_prefill(w: synth.Workload, x: dict, out_f32=False, flags=0, final_z=False, init_z=None,
                force_simt=False, stream=None):
    """Run gla_fwd_ex on generated inputs; returns (out, final_state, final_z) as numpy float64."""
    import torch
    B, H, L, dk, dv = w.B, w.H, w.L, w.dk, w.dv
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    la = to_dev(x["log_alpha"])
    s0 = to_dev(x["init_state"])
    z0 = to_dev(init_z)
    f32in = w.dtype == "f32"
    odt = torch.float32 if (out_f32 or f32in) else torch.bfloat16
    out = torch.full((B, H, L, dv), float("nan"), dtype=odt, device=dev())
    fs = torch.full((B, H, dk, dv), float("nan"), dtype=torch.float32, device=dev())
    fz = torch.full((B, H, dk), float("nan"), dtype=torch.float32, device=dev()) if final_z else None
    fl = flags | (gla.FLAG_FEATURE_ELU1 if w.feature_elu1 else 0) | \
        (gla.FLAG_NORMALIZE if w.normalize else 0) | (gla.FLAG_FORCE_SIMT if force_simt else 0) | \
        (gla.FLAG_SCALAR_GATE if w.scalar_gate else 0)
    st = gla.gla_fwd_ex(q, k, v, out, B, H, L, dk, dv, chunk=w.chunk, log_alpha=la, init_state=s0,
                        init_z=z0, final_state=fs, final_z=fz,
                        in_dtype=gla.F32 if f32in else gla.BF16,
                        out_dtype=gla.F32 if (out_f32 or f32in) else gla.BF16, flags=fl,
                        stream=stream)
    gla.check(st)
    torch.cuda.synchronize()
    _, detail = gla.gla_device_error_detail()
    if detail[0]:
        gla.gla_device_error()
        raise gla.GlaError(f"device wait timed out: {[hex(x) for x in detail]}")
    return (out.float().cpu().numpy().astype(np.float64), fs.cpu().numpy().astype(np.float64),
            None if fz is None else fz.cpu().numpy().astype(np.float64))


def oracle_prefill(w: synth.Workload, x: dict, init_z=None, nthreads=0):
    la = synth.as_f64(x["log_alpha"])
    if w.scalar_gate and la is not None:
        # a per-token gate is the per-channel gate with the same value on every channel
        la = np.repeat(la[..., None], w.dk, axis=-1)
    return oracle.gla_fwd(synth.as_f64(x["q"]), synth.as_f64(x["k"]), synth.as_f64(x["v"]),
                          la, synth.as_f64(x["init_state"]),
                          None if init_z is None else np.asarray(init_z, np.float64),
                          feature_elu1=w.feature_elu1, normalize=w.normalize, nthreads=nthreads)
