"""Failure detection on the boundary, made without faulting a GPU.

- An injected launch failure (GLA_TEST_FAIL_LAUNCH=1): every entry point that
  launches a kernel returns GLA_ERR_CUDA after validating its arguments and
  before any launch (checked on the CPU: the fake pointers are never touched),
  and on the GPU the output buffer stays untouched and the next call works.
- A bounded device wait that runs out: with gla_test_set_waits(limit, stall)
  the prefill kernel's gate role first waits on a barrier that nothing
  completes; after `limit` every role of every CTA stops, drains what it has in
  flight, and the call reports GLA_ERR_TIMEOUT through gla_device_error, with
  the wait's details in gla_device_error_detail.  The device stays usable: the
  next call matches the oracle.
- The error record is one per device, shared by every stream (as gla.h states):
  a timeout in a call on one stream is reported to the next reader on any stream.
"""
import numpy as np
import pytest

import causal_gated_linear_gb300 as gla
import synth

A = 1 << 20  # fake, 16-byte aligned "device" addresses: never dereferenced


@pytest.fixture(scope="module")
def lib():
    gla.build()
    return gla.load()


@pytest.fixture
def inject(monkeypatch):
    monkeypatch.setenv("GLA_TEST_FAIL_LAUNCH", "1")


def test_injected_launch_failure_after_validation(lib, inject):
    # valid arguments: the injected failure
    assert gla.gla_fwd(A, 2 * A, 3 * A, 4 * A, None, 8 * A, None, 1, 1, 64, 64, 64, 64, stream=0) == \
        gla.GLA_ERR_CUDA
    assert gla.gla_decode_step(A, 2 * A, 3 * A, 4 * A, 16 * A, 8 * A, 2, 2, 128, 128, stream=0) == gla.GLA_ERR_CUDA
    assert gla.gla_delta_fwd(A, 2 * A, 3 * A, 4 * A, 8 * A, 1, 1, 64, 64, 64, stream=0) == gla.GLA_ERR_CUDA
    assert gla.gla_bwd(A, 2 * A, 3 * A, 4 * A, 8 * A, 16 * A, 24 * A, 1, 1, 64, 64, 64, stream=0) == \
        gla.GLA_ERR_CUDA
    # invalid arguments are still rejected first, with their own status
    assert gla.gla_fwd(A + 8, 2 * A, 3 * A, 4 * A, None, 8 * A, None, 1, 1, 64, 64, 64, 64, stream=0) == \
        gla.GLA_ERR_MISALIGNED
    assert gla.gla_fwd(A, 2 * A, 3 * A, 4 * A, None, 8 * A, None, 1, 1, 64, 64, 64, 32, stream=0) == \
        gla.GLA_ERR_UNSUPPORTED
    assert gla.gla_decode_step(A, 2 * A, 3 * A, 4 * A, None, 8 * A, 2, 2, 128, 128, stream=0) == \
        gla.GLA_ERR_INVALID


def test_test_hook_is_host_only(lib):
    assert gla.gla_test_set_waits(1000, True) == gla.GLA_OK
    assert gla.gla_test_set_waits(0, False) == gla.GLA_OK


# ---------------------------------------------------------------- GPU

def _prefill(seed, L=600, H=2):
    w = synth.with_shape(synth.PREFILL, B=1, H=H, L=L, init_std=0.1, seed=seed)
    return w, synth.make_prefill(w)


@pytest.mark.gpu
def test_injected_launch_failure_leaves_output_and_device_intact(lib, monkeypatch):
    import torch
    from gpu_util import assert_bf16_close, oracle_prefill, to_dev
    w, x = _prefill(301)
    q, k, v, la, s0 = (to_dev(x[n]) for n in ("q", "k", "v", "log_alpha", "init_state"))
    out = torch.full((1, 2, w.L, w.dv), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    fs = torch.full((1, 2, w.dk, w.dv), float("nan"), device="cuda:0")
    monkeypatch.setenv("GLA_TEST_FAIL_LAUNCH", "1")
    assert gla.gla_fwd(q, k, v, la, s0, out, fs, 1, 2, w.L, w.dk, w.dv, 64) == gla.GLA_ERR_CUDA
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all() and torch.isnan(fs).all()
    monkeypatch.delenv("GLA_TEST_FAIL_LAUNCH")
    gla.check(gla.gla_fwd(q, k, v, la, s0, out, fs, 1, 2, w.L, w.dk, w.dv, 64))
    assert gla.gla_device_error() == gla.GLA_OK
    ro, rs, _ = oracle_prefill(w, x)
    assert_bf16_close(out.float().cpu().numpy(), ro, "out")
    assert_bf16_close(fs.cpu().numpy(), rs, "state")


def _stalled_call(w, x, stream):
    import torch
    from gpu_util import to_dev
    q, k, v, la, s0 = (to_dev(x[n]) for n in ("q", "k", "v", "log_alpha", "init_state"))
    out = torch.empty((1, w.H, w.L, w.dv), dtype=torch.bfloat16, device="cuda:0")
    fs = torch.empty((1, w.H, w.dk, w.dv), device="cuda:0")
    gla.gla_test_set_waits(20_000_000, True)  # 20 ms, then the gate's first wait runs out
    try:
        st = gla.gla_fwd(q, k, v, la, s0, out, fs, 1, w.H, w.L, w.dk, w.dv, 64, stream=stream)
    finally:
        gla.gla_test_set_waits(0, False)
    assert st == gla.GLA_OK  # the launch itself succeeds; the wait runs out on the device
    return q, k, v, la, s0, out, fs


@pytest.mark.gpu
@pytest.mark.parametrize("dvt", ["64", "128"])
def test_wait_that_runs_out_reports_timeout_and_device_recovers(lib, monkeypatch, dvt):
    import torch
    from gpu_util import assert_bf16_close, oracle_prefill
    monkeypatch.setenv("GLA_TC_DVT", dvt)
    assert gla.gla_device_error() == gla.GLA_OK
    w, x = _prefill(302)
    q, k, v, la, s0, out, fs = _stalled_call(w, x, None)
    torch.cuda.synchronize()
    st, detail = gla.gla_device_error_detail()
    assert st == gla.GLA_OK
    assert detail[0] & 1                 # a bounded wait ran out
    # the first wait to run out (the gate's, or another role's waiting on it: all share the limit)
    assert detail[1] & 1 and detail[2] < 768
    assert detail[3] < w.H * (w.dv // int(dvt))  # a CTA of this launch
    assert gla.gla_device_error() == gla.GLA_ERR_TIMEOUT
    assert gla.gla_device_error() == gla.GLA_OK  # read and cleared
    # the same device, the ordinary limit: the call matches the oracle
    gla.check(gla.gla_fwd(q, k, v, la, s0, out, fs, 1, w.H, w.L, w.dk, w.dv, 64))
    assert gla.gla_device_error() == gla.GLA_OK
    ro, rs, _ = oracle_prefill(w, x)
    assert_bf16_close(out.float().cpu().numpy(), ro, "out")
    assert_bf16_close(fs.cpu().numpy(), rs, "state")


@pytest.mark.gpu
def test_error_record_is_shared_by_streams(lib):
    import torch
    from gpu_util import assert_bf16_close, oracle_prefill, to_dev
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    w1, x1 = _prefill(303)
    w2, x2 = _prefill(304, L=300)
    with torch.cuda.stream(s1):
        keep = _stalled_call(w1, x1, s1)  # its buffers stay alive until the stream has drained
    q, k, v, la, s0 = (to_dev(x2[n]) for n in ("q", "k", "v", "log_alpha", "init_state"))
    out = torch.empty((1, 2, w2.L, w2.dv), dtype=torch.bfloat16, device="cuda:0")
    fs = torch.empty((1, 2, w2.dk, w2.dv), device="cuda:0")
    torch.cuda.synchronize()
    gla.check(gla.gla_fwd(q, k, v, la, s0, out, fs, 1, 2, w2.L, w2.dk, w2.dv, 64, stream=s2))
    torch.cuda.synchronize()
    del keep
    # the stream-1 timeout is reported to the first reader, here on stream 2, and cleared there
    assert gla.gla_device_error(s2) == gla.GLA_ERR_TIMEOUT
    assert gla.gla_device_error(s1) == gla.GLA_OK
    ro, rs, _ = oracle_prefill(w2, x2)
    assert_bf16_close(out.float().cpu().numpy(), ro, "stream-2 out")
    assert_bf16_close(fs.cpu().numpy(), rs, "stream-2 state")
