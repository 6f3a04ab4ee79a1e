"""fp64 CPU oracle of causal gated linear attention -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline / reference leg
of `bench.py` may import this package.  The library path never does: it
shares no code with the CUDA kernels and is not a fallback for them.

The arithmetic lives in `gla_oracle.c` (plain C, float64, one token at a
time); this module compiles it with gcc + OpenMP and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict = {}

FEATURE_ELU1 = 1
NORMALIZE = 2


def lib_path(plant: int = 0, build_dir: str | None = None) -> str:
    d = build_dir or _BUILD
    name = "liboracle.so" if plant == 0 else f"liboracle_plant{plant}.so"
    return os.path.join(d, name)


def build(plant: int = 0, build_dir: str | None = None, force: bool = False) -> str:
    """Compile the oracle (or a planted-mistake variant) and return the .so path."""
    out = lib_path(plant, build_dir)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", f"-DORACLE_PLANT={plant}",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(plant: int = 0, build_dir: str | None = None):
    key = (plant, build_dir)
    with _LOCK:
        if key in _LIBS:
            return _LIBS[key]
        lib = ctypes.CDLL(build(plant, build_dir))
        D = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        lib.oracle_gla_fwd.argtypes = [D, D, D, D, D, D, D, D, D, L, L, L, L, L,
                                       ctypes.c_int, ctypes.c_int]
        lib.oracle_gla_fwd.restype = ctypes.c_int
        lib.oracle_gla_decode_step.argtypes = [D, D, D, D, D, D, L, L, L, L, ctypes.c_int]
        lib.oracle_gla_decode_step.restype = ctypes.c_int
        lib.oracle_gla_fwd_chunked.argtypes = [D, D, D, D, D, D, D, L, L, L, L, L, L,
                                               ctypes.c_int]
        lib.oracle_gla_fwd_chunked.restype = ctypes.c_int
        lib.oracle_delta_fwd.argtypes = [D, D, D, D, D, D, D, D, L, L, L, L, ctypes.c_int]
        lib.oracle_delta_fwd.restype = ctypes.c_int
        lib.oracle_gla_bwd.argtypes = [D, D, D, D, D, D, D, D, D, D, D, D, L, L, L, L, ctypes.c_int]
        lib.oracle_gla_bwd.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        _LIBS[key] = lib
        return lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None and a.shape != tuple(shape):
        a = a.reshape(shape)
    return a


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def gla_fwd(q, k, v, log_alpha=None, init_state=None, init_z=None, feature_elu1=False,
            normalize=False, nthreads=0, plant=0, build_dir=None):
    """Token-by-token recurrence.  q, k: [..., L, dk]; v: [..., L, dv].

    Leading dims are flattened into (batch*head).  Returns (out, final_state,
    final_z) as float64 arrays; final_z is None unless `normalize`.
    """
    q = _f64(q)
    lead = q.shape[:-2]
    L, dk = q.shape[-2:]
    dv = np.shape(v)[-1]
    BH = int(np.prod(lead)) if lead else 1
    q = q.reshape(BH, L, dk)
    k = _f64(k).reshape(BH, L, dk)
    v = _f64(v).reshape(BH, L, dv)
    la = _f64(log_alpha).reshape(BH, L, dk) if log_alpha is not None else None
    s0 = _f64(init_state).reshape(BH, dk, dv) if init_state is not None else None
    z0 = _f64(init_z).reshape(BH, dk) if init_z is not None else None
    out = np.empty((BH, L, dv), dtype=np.float64)
    fs = np.empty((BH, dk, dv), dtype=np.float64)
    fz = np.empty((BH, dk), dtype=np.float64) if normalize else None
    flags = (FEATURE_ELU1 if feature_elu1 else 0) | (NORMALIZE if normalize else 0)
    rc = _load(plant, build_dir).oracle_gla_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(s0), _ptr(z0), _ptr(out), _ptr(fs), _ptr(fz),
        1, BH, L, dk, dv, flags, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gla_fwd failed ({rc})")
    out = out.reshape(*lead, L, dv)
    fs = fs.reshape(*lead, dk, dv)
    if fz is not None:
        fz = fz.reshape(*lead, dk)
    return out, fs, fz


def gla_fwd_chunked(q, k, v, log_alpha=None, init_state=None, chunk=64, nthreads=0):
    """Chunk-wise restatement of the same function (fp64)."""
    q = _f64(q)
    lead = q.shape[:-2]
    L, dk = q.shape[-2:]
    dv = np.shape(v)[-1]
    BH = int(np.prod(lead)) if lead else 1
    q = q.reshape(BH, L, dk)
    k = _f64(k).reshape(BH, L, dk)
    v = _f64(v).reshape(BH, L, dv)
    la = _f64(log_alpha).reshape(BH, L, dk) if log_alpha is not None else None
    s0 = _f64(init_state).reshape(BH, dk, dv) if init_state is not None else None
    out = np.empty((BH, L, dv), dtype=np.float64)
    fs = np.empty((BH, dk, dv), dtype=np.float64)
    rc = _load().oracle_gla_fwd_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(s0), _ptr(out),
                                        _ptr(fs), 1, BH, L, dk, dv, int(chunk), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gla_fwd_chunked failed ({rc})")
    return out.reshape(*lead, L, dv), fs.reshape(*lead, dk, dv)


def gla_decode_step(q, k, v, log_alpha, state, nthreads=0, plant=0, build_dir=None):
    """One decode step.  q, k, log_alpha [..., dk]; v [..., dv]; state [..., dk, dv].

    Returns (out, new_state); the input `state` array is not modified.
    """
    q = _f64(q)
    lead = q.shape[:-1]
    dk = q.shape[-1]
    dv = np.shape(v)[-1]
    n = int(np.prod(lead)) if lead else 1
    st = np.array(state, dtype=np.float64, copy=True).reshape(n, dk, dv)
    out = np.empty((n, dv), dtype=np.float64)
    la = _f64(log_alpha).reshape(n, dk) if log_alpha is not None else None
    rc = _load(plant, build_dir).oracle_gla_decode_step(
        _ptr(q.reshape(n, dk)), _ptr(_f64(k).reshape(n, dk)), _ptr(_f64(v).reshape(n, dv)),
        _ptr(la), _ptr(st), _ptr(out), 1, n, dk, dv, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gla_decode_step failed ({rc})")
    return out.reshape(*lead, dv), st.reshape(*lead, dk, dv)


def delta_fwd(q, k, v, beta, log_alpha=None, init_state=None, nthreads=0, plant=0, build_dir=None):
    """Delta rule, token by token ("linear-attention" blog, Delta attention; gated when
    log_alpha is given).  q, k, log_alpha: [..., L, dk]; v: [..., L, dv]; beta: [..., L].

    Returns (out, final_state) as float64 arrays.
    """
    q = _f64(q)
    lead = q.shape[:-2]
    L, dk = q.shape[-2:]
    dv = np.shape(v)[-1]
    BH = int(np.prod(lead)) if lead else 1
    q = q.reshape(BH, L, dk)
    k = _f64(k).reshape(BH, L, dk)
    v = _f64(v).reshape(BH, L, dv)
    b = _f64(beta).reshape(BH, L)
    la = _f64(log_alpha).reshape(BH, L, dk) if log_alpha is not None else None
    s0 = _f64(init_state).reshape(BH, dk, dv) if init_state is not None else None
    out = np.empty((BH, L, dv), dtype=np.float64)
    fs = np.empty((BH, dk, dv), dtype=np.float64)
    rc = _load(plant, build_dir).oracle_delta_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(la), _ptr(s0),
                                                  _ptr(out), _ptr(fs), BH, L, dk, dv, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_delta_fwd failed ({rc})")
    return out.reshape(*lead, L, dv), fs.reshape(*lead, dk, dv)


def gla_bwd(q, k, v, dout, log_alpha=None, init_state=None, dfinal=None, nthreads=0, plant=0,
            build_dir=None):
    """Reverse mode of the recurrence ("Gated Linear Attention", GLA Recurrent Form).
    q, k, log_alpha: [..., L, dk]; v, dout: [..., L, dv]; init_state, dfinal: [..., dk, dv].

    Returns (dq, dk, dv, dlog_alpha or None, dinit) as float64 arrays.  Keeps every state:
    memory L * dk * dv doubles per head.
    """
    q = _f64(q)
    lead = q.shape[:-2]
    L, dk = q.shape[-2:]
    dv = np.shape(v)[-1]
    BH = int(np.prod(lead)) if lead else 1
    q = q.reshape(BH, L, dk)
    k = _f64(k).reshape(BH, L, dk)
    v = _f64(v).reshape(BH, L, dv)
    do = _f64(dout).reshape(BH, L, dv)
    la = _f64(log_alpha).reshape(BH, L, dk) if log_alpha is not None else None
    s0 = _f64(init_state).reshape(BH, dk, dv) if init_state is not None else None
    df = _f64(dfinal).reshape(BH, dk, dv) if dfinal is not None else None
    dq = np.empty((BH, L, dk))
    dkk = np.empty((BH, L, dk))
    dvv = np.empty((BH, L, dv))
    dla = np.empty((BH, L, dk)) if la is not None else None
    dinit = np.empty((BH, dk, dv))
    rc = _load(plant, build_dir).oracle_gla_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(s0), _ptr(do),
                                                _ptr(df), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dla),
                                                _ptr(dinit), BH, L, dk, dv, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gla_bwd failed ({rc})")
    r = lambda a, *s: None if a is None else a.reshape(*lead, *s)
    return r(dq, L, dk), r(dkk, L, dk), r(dvv, L, dv), r(dla, L, dk), r(dinit, dk, dv)
