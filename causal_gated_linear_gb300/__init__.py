"""Python binding of the GB300 causal gated-linear-attention library (libgla.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI (include/gla.h).  PyTorch provides device memory and
streams.  There is no CPU or PyTorch fallback: if the shared library has not
been built, importing the functions raises.

The functions mirror the C entry points:

    gla_fwd(q, k, v, log_alpha, init_state, out, final_state,
            B, H, L, dk, dv, chunk, stream=None) -> int status
    gla_fwd_ex(q, k, v, out, B, H, L, dk, dv, chunk=64, log_alpha=None,
               init_state=None, init_z=None, final_state=None, final_z=None,
               in_dtype=BF16, out_dtype=BF16, flags=0, stream=None) -> int
    gla_fwd_host(host, dev, B, H, L, dk, dv, chunk=64, groups=4, in_dtype=BF16,
                 out_dtype=BF16, flags=0, copy_in=None, compute=None, copy_out=None) -> int
    gla_decode_step(q, k, v, log_alpha, state, out, B, H, dk, dv, stream=None)
    gla_delta_fwd(q, k, v, beta, out, B, H, L, dk, dv, log_alpha=None, init_state=None,
                  final_state=None, out_dtype=BF16, stream=None) -> int
    gla_bwd(q, k, v, dout, dq, dk, dv, B, H, L, dk_dim, dv_dim, log_alpha=None, init_state=None,
            dfinal=None, dlog_alpha=None, dinit=None, in_dtype=BF16, flags=0, stream=None) -> int
    gla_device_error(stream=None) -> int
    gla_test_set_waits(limit_ns=0, stall=False) -> int   (test only)
    gla_status_string(status) -> str
    gla_version() -> str

Tensor arguments may be torch tensors (their data_ptr is passed), raw ints
(device addresses) or None (NULL).  `stream` defaults to torch's current
stream.  A non-zero status is returned as is; `check(status)` raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

GLA_OK, GLA_ERR_INVALID, GLA_ERR_UNSUPPORTED, GLA_ERR_MISALIGNED, GLA_ERR_CUDA, GLA_ERR_TIMEOUT = range(6)
BF16, F32 = 0, 1
FLAG_FEATURE_ELU1, FLAG_NORMALIZE, FLAG_FORCE_SIMT, FLAG_FORCE_CHUNK, FLAG_SCALAR_GATE = 1, 2, 4, 8, 16

EXPORTED = ["gla_fwd", "gla_fwd_ex", "gla_fwd_host", "gla_decode_step", "gla_delta_fwd", "gla_delta_fwd_ex", "gla_bwd",
            "gla_device_error",
            "gla_device_error_detail", "gla_test_set_waits", "gla_status_string", "gla_version"]


class GlaError(RuntimeError):
    pass


class _FwdArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("log_alpha", ctypes.c_void_p), ("init_state", ctypes.c_void_p),
                ("init_z", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("final_state", ctypes.c_void_p), ("final_z", ctypes.c_void_p),
                ("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("flags", ctypes.c_uint)]


_LIB = None


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libgla.so (built in-tree by `build()`); raises if it is missing."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or _build.LIB
    if not os.path.exists(p):
        raise GlaError(f"libgla.so not built ({p}); run causal_gated_linear_gb300.build()")
    lib = ctypes.CDLL(p)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.gla_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
    lib.gla_fwd.restype = i
    lib.gla_fwd_ex.argtypes = [ctypes.POINTER(_FwdArgs), vp]
    lib.gla_fwd_ex.restype = i
    lib.gla_fwd_host.argtypes = [ctypes.POINTER(_FwdArgs), ctypes.POINTER(_FwdArgs), i, vp, vp, vp]
    lib.gla_fwd_host.restype = i
    lib.gla_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, vp]
    lib.gla_decode_step.restype = i
    lib.gla_delta_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
    lib.gla_delta_fwd.restype = i
    lib.gla_delta_fwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_uint, vp]
    lib.gla_delta_fwd_ex.restype = i
    lib.gla_bwd.argtypes = [vp] * 12 + [i] * 6 + [ctypes.c_uint, vp]
    lib.gla_bwd.restype = i
    lib.gla_device_error.argtypes = [vp]
    lib.gla_device_error.restype = i
    lib.gla_device_error_detail.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.gla_device_error_detail.restype = i
    lib.gla_test_set_waits.argtypes = [ctypes.c_ulonglong, i]
    lib.gla_test_set_waits.restype = i
    lib.gla_status_string.argtypes = [i]
    lib.gla_status_string.restype = ctypes.c_char_p
    lib.gla_version.argtypes = []
    lib.gla_version.restype = ctypes.c_char_p
    if path is None:
        _LIB = lib
    return lib


def build(force: bool = False) -> str:
    """Compile libgla.so for sm_103a in-tree and load it."""
    p = _build.build(force=force)
    global _LIB
    _LIB = None
    load()
    return p


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(status: int) -> None:
    if status != GLA_OK:
        raise GlaError(gla_status_string(status))


def gla_fwd(q, k, v, log_alpha, init_state, out, final_state, B, H, L, dk, dv, chunk=64,
            stream=None) -> int:
    return load().gla_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(init_state), _ptr(out),
                          _ptr(final_state), B, H, L, dk, dv, chunk, _stream(stream))


def gla_fwd_ex(q, k, v, out, B, H, L, dk, dv, chunk=64, log_alpha=None, init_state=None,
               init_z=None, final_state=None, final_z=None, in_dtype=BF16, out_dtype=BF16, flags=0,
               stream=None) -> int:
    a = _FwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(init_state), _ptr(init_z),
                 _ptr(out), _ptr(final_state), _ptr(final_z), B, H, L, dk, dv, chunk, in_dtype,
                 out_dtype, flags)
    return load().gla_fwd_ex(ctypes.byref(a), _stream(stream))


def gla_fwd_host(host: dict, dev: dict, B, H, L, dk, dv, chunk=64, groups=4, in_dtype=BF16, out_dtype=BF16,
                 flags=0, copy_in=None, compute=None, copy_out=None) -> int:
    """`host` and `dev` map gla_fwd_args field names (q, k, v, log_alpha, init_state, init_z, out,
    final_state, final_z) to host (pinned) and device tensors; missing names are NULL."""
    names = ("q", "k", "v", "log_alpha", "init_state", "init_z", "out", "final_state", "final_z")

    def args(m):
        return _FwdArgs(*(_ptr(m.get(n)) for n in names), B, H, L, dk, dv, chunk, in_dtype, out_dtype, flags)

    ha, da = args(host), args(dev)
    return load().gla_fwd_host(ctypes.byref(ha), ctypes.byref(da), groups, _stream(copy_in), _stream(compute),
                               _stream(copy_out))


def gla_decode_step(q, k, v, log_alpha, state, out, B, H, dk, dv, stream=None) -> int:
    return load().gla_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(state),
                                  _ptr(out), B, H, dk, dv, _stream(stream))


def gla_delta_fwd(q, k, v, beta, out, B, H, L, dk, dv, log_alpha=None, init_state=None, final_state=None,
                  out_dtype=BF16, flags=0, stream=None) -> int:
    """The delta rule; `flags` (GLA_FLAG_FORCE_SIMT) goes through gla_delta_fwd_ex."""
    if flags:
        return load().gla_delta_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_alpha), _ptr(init_state),
                                       _ptr(out), _ptr(final_state), B, H, L, dk, dv, out_dtype, flags,
                                       _stream(stream))
    return load().gla_delta_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_alpha), _ptr(init_state),
                                _ptr(out), _ptr(final_state), B, H, L, dk, dv, out_dtype, _stream(stream))


def gla_bwd(q, k, v, dout, dq, dk, dv, B, H, L, dk_dim, dv_dim, log_alpha=None, init_state=None, dfinal=None,
            dlog_alpha=None, dinit=None, in_dtype=BF16, flags=0, stream=None) -> int:
    return load().gla_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(init_state), _ptr(dout), _ptr(dfinal),
                          _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dlog_alpha), _ptr(dinit), B, H, L, dk_dim, dv_dim,
                          in_dtype, flags, _stream(stream))


def gla_device_error(stream=None) -> int:
    return load().gla_device_error(_stream(stream))


def gla_device_error_detail(stream=None):
    """(status, [flags, first wait, thread, cta]) of the device error record (not cleared)."""
    buf = (ctypes.c_uint * 4)()
    st = load().gla_device_error_detail(_stream(stream), buf)
    return st, list(buf)


def gla_test_set_waits(limit_ns: int = 0, stall: bool = False) -> int:
    """Test only: limit of the prefill kernel's pipeline waits for later calls (0: the 2 s default),
    and whether its gate role first waits on a barrier that nothing completes."""
    return load().gla_test_set_waits(int(limit_ns), 1 if stall else 0)


def gla_status_string(status: int) -> str:
    return load().gla_status_string(int(status)).decode()


def gla_version() -> str:
    return load().gla_version().decode()
