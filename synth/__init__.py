"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the attention method itself.  It only
draws numbers and rounds them to the storage types the library consumes:

* a counter-based generator (splitmix64 of a per-tensor key plus the element
  index), so any element of any tensor can be regenerated on its own;
* Box-Muller normals from the two 32-bit halves of one 64-bit draw;
* round-to-nearest-even casts float64 -> float32 -> bfloat16;
* the gate input recipe log(alpha) = logsigmoid(g) / temperature, which is how
  the workloads below describe their *inputs* (the library takes log(alpha)
  directly; the gate projection that would produce g is not part of the path).

Workload recipes (shapes and distributions) follow the five configurations
the library is measured on: fp32 GLA (B1 H1 L256 d32), elu+1 normalised
linear attention (B4 H8 L2048 d64), GLA prefill (B8 H16 L4096 d128),
long-context GLA prefill (B1 H32 L65536 dk128 dv256, nonzero initial state)
and the decode step (256 sequences x H32, d128, 1024 steps).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)

# tensor ids (the "tensor" part of the counter key)
T_Q, T_K, T_V, T_G, T_S0, T_BETA, T_DOUT, T_DFIN = 1, 2, 3, 4, 5, 6, 7, 8

BASE_SEED = 20261202


def _splitmix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser applied to x + golden gamma (uint64, wraps mod 2^64)."""
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        return z ^ (z >> np.uint64(31))


def tensor_key(seed: int, tensor_id: int, step: int = 0) -> np.uint64:
    k = np.array([((seed * 0x100000001B3) ^ (tensor_id << 40) ^ (step << 8)) & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    return _splitmix64(_splitmix64(k))[0]


def _normal_block(key: np.uint64, start: int, n: int) -> np.ndarray:
    idx = np.arange(start, start + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = _splitmix64(idx + key)
    hi = (x >> np.uint64(32)).astype(np.float64)
    lo = (x & np.uint64(0xFFFFFFFF)).astype(np.float64)
    u1 = (hi + 0.5) * (1.0 / 4294967296.0)
    u2 = (lo + 0.5) * (1.0 / 4294967296.0)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos((2.0 * math.pi) * u2)


_POOL = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def normals(seed: int, tensor_id: int, shape, step: int = 0, start: int = 0,
            mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """float64 N(mean, std) array; element e is a pure function of (seed, tensor, step, start+e)."""
    n = int(np.prod(shape))
    key = tensor_key(seed, tensor_id, step)
    block = 1 << 22
    if n <= block:
        out = _normal_block(key, start, n)
    else:
        out = np.empty(n, dtype=np.float64)

        def work(s):
            e = min(n, s + block)
            out[s:e] = _normal_block(key, start + s, e - s)

        list(_pool().map(work, range(0, n, block)))
    if std != 1.0:
        out *= std
    if mean != 0.0:
        out += mean
    return out.reshape(shape)


def to_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32)


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        r = (u + rounding) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 (RNE)."""
    return f32_to_bf16_bits(to_f32(x))


def log_sigmoid(g: np.ndarray) -> np.ndarray:
    """Numerically safe log(sigmoid(g)) in float64 (input recipe for log alpha)."""
    return np.minimum(g, 0.0) - np.log1p(np.exp(-np.abs(g)))


# --------------------------------------------------------------------------- recipes


@dataclass
class Workload:
    name: str
    B: int
    H: int
    L: int
    dk: int
    dv: int
    chunk: int = 64
    dtype: str = "bf16"          # storage type of q, k, v (and out for prefill)
    gate: bool = True            # log alpha present
    gate_mean: float = 4.0
    gate_std: float = 1.5
    gate_temp: float = 16.0      # log alpha = logsigmoid(g) / gate_temp
    qk_scale: bool = True        # q, k multiplied by dk^-1/2 at generation
    feature_elu1: bool = False
    normalize: bool = False
    scalar_gate: bool = False    # log alpha [B,H,L]: one gate per token, shared by the channels
    init_std: float = 0.0        # 0 -> zero initial state
    seed: int = BASE_SEED
    extra: dict = field(default_factory=dict)


# fp32 SIMT path: B1 H1 L256 dk = dv = 32, gate logsigmoid(N(3, 1))
FP32_SMALL = Workload("gla_fp32_B1H1L256d32", 1, 1, 256, 32, 32, dtype="f32",
                      gate_mean=3.0, gate_std=1.0, gate_temp=1.0, seed=BASE_SEED + 0)
# plain causal linear attention with phi = elu + 1 and the normaliser: B4 H8 L2048 d64
ELU_NORM = Workload("linattn_elu1_norm_B4H8L2048d64", 4, 8, 2048, 64, 64, gate=False,
                    qk_scale=False, feature_elu1=True, normalize=True, seed=BASE_SEED + 1)
# gated prefill: B8 H16 L4096 dk = dv = 128, bf16
PREFILL = Workload("gla_prefill_B8H16L4096d128", 8, 16, 4096, 128, 128, seed=BASE_SEED + 2)
# long-context gated prefill with an initial state: B1 H32 L65536 dk128 dv256, bf16
LONGCTX = Workload("gla_longctx_B1H32L65536dk128dv256", 1, 32, 65536, 128, 256,
                   init_std=0.1, seed=BASE_SEED + 3)
PREFILL_WORKLOADS = (FP32_SMALL, ELU_NORM, PREFILL, LONGCTX)

# several new tokens per sequence on top of a decode-sized state (the prefill -> decode
# hand-off): decode distributions (q, k, v ~ N(0,1), log alpha = logsigmoid(N(4, 1.5)),
# S ~ N(0, 0.1)), 8 tokens per call
DECODE_MULTI = Workload("gla_decode_multi_256seqH32d128T8", 256, 32, 8, 128, 128, qk_scale=False,
                        gate_temp=1.0, init_std=0.1, seed=BASE_SEED + 5)

DECODE = dict(name="gla_decode_256seqH32d128x1024", NS=256, H=32, dk=128, dv=128, steps=1024,
              gate_mean=4.0, gate_std=1.5, state_std=0.1, seed=BASE_SEED + 4)


def with_shape(w: Workload, **kw) -> Workload:
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


def make_prefill(w: Workload, heads=None):
    """Inputs of a prefill workload as host arrays.

    Returns a dict with q, k, v (uint16 bf16 bits or float32, shape [B,H,L,d]),
    log_alpha (float32 [B,H,L,dk] or None) and init_state (float32 [B,H,dk,dv]
    or None).  `heads`, if given, is a list of flat (b*H+h) indices and only
    those heads are generated (same values as in the full tensors).
    """
    B, H, L, dk, dv = w.B, w.H, w.L, w.dk, w.dv
    sel = list(range(B * H)) if heads is None else list(heads)

    def gen(tid, d, std=1.0, mean=0.0):
        per = L * d
        parts = [normals(w.seed, tid, (L, d), start=hh * per, mean=mean, std=std) for hh in sel] \
            if heads is not None else [normals(w.seed, tid, (B * H * L * d,), mean=mean, std=std)]
        return np.concatenate([p.reshape(-1) for p in parts])

    qs = 1.0 / math.sqrt(dk) if w.qk_scale else 1.0
    q = gen(T_Q, dk, std=qs)
    k = gen(T_K, dk, std=qs)
    v = gen(T_V, dv)
    nh = len(sel)
    shp_k = (nh, L, dk) if heads is not None else (B, H, L, dk)
    shp_v = (nh, L, dv) if heads is not None else (B, H, L, dv)
    if w.dtype == "bf16":
        q, k, v = to_bf16_bits(q), to_bf16_bits(k), to_bf16_bits(v)
    else:
        q, k, v = to_f32(q), to_f32(k), to_f32(v)
    out = dict(q=q.reshape(shp_k), k=k.reshape(shp_k), v=v.reshape(shp_v), log_alpha=None,
               init_state=None)
    if w.gate:
        out["log_alpha"] = gate_log_alpha(w, heads)
    if w.init_std > 0:
        per = dk * dv
        if heads is not None:
            s0 = np.concatenate([normals(w.seed, T_S0, (per,), start=hh * per, std=w.init_std)
                                 for hh in sel])
            out["init_state"] = to_f32(s0).reshape(nh, dk, dv)
        else:
            out["init_state"] = to_f32(normals(w.seed, T_S0, (B * H * per,), std=w.init_std)
                                       ).reshape(B, H, dk, dv)
    return out


def gate_log_alpha(w: Workload, heads=None):
    """log alpha of a gated prefill workload, float32 [B,H,L,dk] ([B,H,L] with scalar_gate);
    the values make_prefill returns for it."""
    B, H, L, dk = w.B, w.H, w.L, w.dk
    sel = list(range(B * H)) if heads is None else list(heads)
    gd = 1 if w.scalar_gate else dk
    per = L * gd
    if heads is None:
        g = normals(w.seed, T_G, (B * H * per,), mean=w.gate_mean, std=w.gate_std)
    else:
        g = np.concatenate([normals(w.seed, T_G, (per,), start=hh * per, mean=w.gate_mean, std=w.gate_std)
                            for hh in sel])
    lead = (len(sel),) if heads is not None else (B, H)
    shp = lead + ((L,) if w.scalar_gate else (L, dk))
    return to_f32(log_sigmoid(g) / w.gate_temp).reshape(shp)


# delta-rule workload: the B8 H16 L4096 d128 prefill shape; q and k rows of unit length,
# v ~ N(0,1), beta = sigmoid(N(0,1)) per token, the prefill gate (logsigmoid(N(4, 1.5)) / 16)
DELTA = Workload("gla_delta_B8H16L4096d128", 8, 16, 4096, 128, 128, qk_scale=False,
                 seed=BASE_SEED + 6)


def make_delta(w: Workload, heads=None):
    """Inputs of a delta-rule workload: q, k (rows scaled to unit length, then bf16 bits),
    v (bf16 bits), beta float32 [.., L], log_alpha float32 [.., L, dk] or None, init_state
    float32 or None.  `heads` selects flat (b*H+h) indices, as in make_prefill."""
    x = make_prefill(w, heads)
    B, H, L, dk = w.B, w.H, w.L, w.dk
    sel = list(range(B * H)) if heads is None else list(heads)
    for n, tid in (("q", T_Q), ("k", T_K)):
        parts = [normals(w.seed, tid, (L, dk), start=hh * L * dk) for hh in sel] if heads is not None \
            else [normals(w.seed, tid, (B * H * L * dk,))]
        a = np.concatenate([p.reshape(-1) for p in parts]).reshape(-1, dk)
        a = a / np.linalg.norm(a, axis=1, keepdims=True)
        x[n] = to_bf16_bits(a).reshape(x[n].shape)
    bparts = [normals(w.seed, T_BETA, (L,), start=hh * L) for hh in sel] if heads is not None \
        else [normals(w.seed, T_BETA, (B * H * L,))]
    g = np.concatenate([p.reshape(-1) for p in bparts])
    lead = (len(sel),) if heads is not None else (B, H)
    x["beta"] = to_f32(1.0 / (1.0 + np.exp(-g))).reshape(lead + (L,))
    return x


# backward workload: the gated prefill (B8 H16 L4096 dk = dv = 128, bf16, its gate
# and q/k scale) with an output gradient dout ~ N(0, 1) per element
BWD = Workload("gla_bwd_B8H16L4096d128", 8, 16, 4096, 128, 128, seed=BASE_SEED + 7)


def make_bwd(w: Workload, heads=None, dfinal_std=0.0):
    """Inputs of a backward workload: make_prefill's, plus dout (bf16 bits or float32, like v)
    and dfinal (float32 [.., dk, dv] ~ N(0, dfinal_std), or None when dfinal_std == 0)."""
    x = make_prefill(w, heads)
    B, H, L, dk, dv = w.B, w.H, w.L, w.dk, w.dv
    sel = list(range(B * H)) if heads is None else list(heads)
    lead = (len(sel),) if heads is not None else (B, H)
    parts = [normals(w.seed, T_DOUT, (L * dv,), start=hh * L * dv) for hh in sel] if heads is not None \
        else [normals(w.seed, T_DOUT, (B * H * L * dv,))]
    d = np.concatenate([p.reshape(-1) for p in parts])
    x["dout"] = (to_bf16_bits(d) if w.dtype == "bf16" else to_f32(d)).reshape(lead + (L, dv))
    x["dfinal"] = None
    if dfinal_std > 0:
        per = dk * dv
        parts = [normals(w.seed, T_DFIN, (per,), start=hh * per, std=dfinal_std) for hh in sel] \
            if heads is not None else [normals(w.seed, T_DFIN, (B * H * per,), std=dfinal_std)]
        x["dfinal"] = to_f32(np.concatenate([p.reshape(-1) for p in parts])).reshape(lead + (dk, dv))
    return x


def decode_state(NS, H, dk, dv, std, seed, heads=None):
    per = dk * dv
    if heads is None:
        return to_f32(normals(seed, T_S0, (NS * H * per,), std=std)).reshape(NS, H, dk, dv)
    return to_f32(np.concatenate([normals(seed, T_S0, (per,), start=hh * per, std=std)
                                  for hh in heads])).reshape(len(heads), dk, dv)


def decode_token(NS, H, dk, dv, step, seed, gate_mean=4.0, gate_std=1.5, heads=None):
    """One decode step's token for every (sequence, head): q,k,v bf16 bits, log alpha f32."""
    def gen(tid, d, mean=0.0, std=1.0):
        if heads is None:
            return normals(seed, tid, (NS * H * d,), step=step + 1, mean=mean, std=std)
        return np.concatenate([normals(seed, tid, (d,), step=step + 1, start=hh * d,
                                       mean=mean, std=std) for hh in heads])
    shp_k = (NS, H, dk) if heads is None else (len(heads), dk)
    shp_v = (NS, H, dv) if heads is None else (len(heads), dv)
    q = to_bf16_bits(gen(T_Q, dk)).reshape(shp_k)
    k = to_bf16_bits(gen(T_K, dk)).reshape(shp_k)
    v = to_bf16_bits(gen(T_V, dv)).reshape(shp_v)
    la = to_f32(log_sigmoid(gen(T_G, dk, mean=gate_mean, std=gate_std))).reshape(shp_k)
    return dict(q=q, k=k, v=v, log_alpha=la)


def as_f64(x):
    """Exact float64 view of a generated array (bf16 bits or float32)."""
    if x is None:
        return None
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float64)
