"""The C-ABI library loads, exports what include/gla.h declares, and rejects
bad arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

import causal_gated_linear_gb300 as gla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gla.build()
    return gla.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "gla.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(gla_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert set(gla.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert "sm_103a" in gla.gla_version()
    assert gla.gla_status_string(0) == "GLA_OK"
    assert gla.gla_status_string(5) == "GLA_ERR_TIMEOUT"
    assert gla.gla_status_string(99) == "GLA_ERR_UNKNOWN"


A = 1 << 20  # fake, 16-byte aligned "device" addresses: never dereferenced


def _fwd(**kw):
    base = dict(q=A, k=2 * A, v=3 * A, log_alpha=4 * A, init_state=None, out=8 * A,
                final_state=None, B=1, H=1, L=64, dk=64, dv=64, chunk=64)
    base.update(kw)
    return gla.gla_fwd(base["q"], base["k"], base["v"], base["log_alpha"], base["init_state"],
                       base["out"], base["final_state"], base["B"], base["H"], base["L"], base["dk"],
                       base["dv"], base["chunk"], stream=0)


@pytest.mark.parametrize("kw,status", [
    (dict(chunk=32), gla.GLA_ERR_UNSUPPORTED),
    (dict(dk=300), gla.GLA_ERR_UNSUPPORTED),
    (dict(B=0), gla.GLA_ERR_INVALID),
    (dict(H=-1), gla.GLA_ERR_INVALID),
    (dict(L=-5), gla.GLA_ERR_INVALID),
    (dict(q=None), gla.GLA_ERR_INVALID),
    (dict(out=None), gla.GLA_ERR_INVALID),
    (dict(q=A + 8), gla.GLA_ERR_MISALIGNED),
    (dict(log_alpha=4 * A + 4), gla.GLA_ERR_MISALIGNED),
    (dict(out=A), gla.GLA_ERR_INVALID),                 # out aliases q
    (dict(out=3 * A + 64), gla.GLA_ERR_INVALID),        # out overlaps v
    (dict(init_state=16 * A, final_state=16 * A + 256), gla.GLA_ERR_INVALID),  # partial alias
])
def test_prefill_validation(lib, kw, status):
    assert _fwd(**kw) == status


def test_prefill_ex_validation(lib):
    assert gla.gla_fwd_ex(A, 2 * A, 3 * A, 8 * A, 1, 1, 64, 64, 64, in_dtype=7, stream=0) == \
        gla.GLA_ERR_INVALID
    assert gla.gla_fwd_ex(A, 2 * A, 3 * A, 8 * A, 1, 1, 64, 64, 64, flags=1 << 5, stream=0) == \
        gla.GLA_ERR_INVALID
    assert gla.gla_fwd_ex(A, 2 * A, 3 * A, 8 * A, 1, 1, 64, 64, 64, chunk=128, stream=0) == \
        gla.GLA_ERR_UNSUPPORTED


def _dec(**kw):
    base = dict(q=A, k=2 * A, v=3 * A, log_alpha=4 * A, state=16 * A, out=8 * A, B=2, H=2, dk=128,
                dv=128)
    base.update(kw)
    return gla.gla_decode_step(base["q"], base["k"], base["v"], base["log_alpha"], base["state"],
                               base["out"], base["B"], base["H"], base["dk"], base["dv"], stream=0)


@pytest.mark.parametrize("kw,status", [
    (dict(dv=6), gla.GLA_ERR_UNSUPPORTED),
    (dict(dv=1024), gla.GLA_ERR_UNSUPPORTED),
    (dict(dk=600), gla.GLA_ERR_UNSUPPORTED),
    (dict(B=0), gla.GLA_ERR_INVALID),
    (dict(state=None), gla.GLA_ERR_INVALID),
    (dict(state=16 * A + 4), gla.GLA_ERR_MISALIGNED),
    (dict(out=16 * A + 1024), gla.GLA_ERR_INVALID),     # out inside the state
])
def test_decode_validation(lib, kw, status):
    assert _dec(**kw) == status


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(gla.GlaError):
        gla.load(str(tmp_path / "nope.so"))
