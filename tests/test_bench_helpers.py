"""CPU checks of the benchmark's own arithmetic: the algorithmic bytes and
flops behind every roofline, the throughput formula, the clock-sample window
and the kernel-source hash that guards the recorded DRAM traffic."""
import os
import shutil
import time

import bench
import synth


def test_prefill_bytes_and_flops_long_context():
    # 32 heads x (65536 tokens x (q 256 + k 256 + v 512 + log alpha 512 + out 512 bytes)
    #             + initial and final fp32 state 2 x 128 x 256 x 4 bytes)
    assert bench.prefill_bytes(synth.LONGCTX) == 32 * (65536 * 2048 + 2 * 128 * 256 * 4) == 4303355904
    # 2 L C (dk + dv) intra-chunk + 4 L dk dv state products, per head
    assert bench.prefill_flops(synth.LONGCTX) == 32 * (2 * 65536 * 64 * 384 + 4 * 65536 * 128 * 256)


def test_prefill_bytes_per_token_gate_and_no_initial_state():
    w = synth.with_shape(synth.LONGCTX, scalar_gate=True, init_std=0.0)
    assert bench.prefill_bytes(w) == 32 * (65536 * (256 + 256 + 512 + 4 + 512) + 128 * 256 * 4)


def test_decode_bytes():
    # 8192 heads x (state in + out 2 x 64 KB, q, k bf16, v bf16, log alpha fp32, out fp32)
    assert bench.decode_bytes(256, 32, 128, 128) == 8192 * (131072 + 256 + 256 + 256 + 512 + 512) == 1088421888
    assert bench.decode_multi_bytes(synth.DECODE_MULTI) == 8192 * (131072 + 8 * (512 + 256 + 512 + 256))


def test_alu_flop_counts():
    assert bench.delta_flops(synth.DELTA) == 128 * 4096 * 7 * 128 * 128
    assert bench.bwd_flops(synth.BWD) == 128 * 4096 * 15 * 128 * 128
    assert bench.bwd_flops(synth.with_shape(synth.BWD, gate=False)) == 128 * 4096 * 12 * 128 * 128


def test_job_throughput_is_all_ranks_over_slowest():
    assert bench.job_throughput(65536, 10, 4, 20.0) == 65536 * 10 * 4 / 0.02


def test_source_hash_ignores_comments_only(tmp_path):
    src = os.path.join(bench.ROOT, "causal_gated_linear_gb300", "csrc")
    for f in bench.KERNEL_SOURCES["gla_decode_kernel"]:
        shutil.copy(os.path.join(src, f), tmp_path / f)
    h0 = bench.kernel_source_hash("gla_decode_kernel", str(tmp_path))
    assert h0 == bench.kernel_source_hash("gla_decode_kernel")
    p = tmp_path / bench.KERNEL_SOURCES["gla_decode_kernel"][0]
    p.write_text("// a new comment\n/* and a block\n comment */\n" + p.read_text().replace("\n", "\n\n"))
    assert bench.kernel_source_hash("gla_decode_kernel", str(tmp_path)) == h0
    p.write_text(p.read_text().replace("kUnroll = 8", "kUnroll = 4"))
    assert bench.kernel_source_hash("gla_decode_kernel", str(tmp_path)) != h0


def test_clock_samples_outside_the_timed_region_are_dropped(tmp_path, monkeypatch):
    monkeypatch.setenv("GLA_BENCH_CLOCKS_DIR", str(tmp_path))
    c = bench.ClockSampler(0)
    c.proc = object()  # as if nvidia-smi had run
    rows = ["2026/12/03 01:50:09.100, 0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
            "2026/12/03 01:50:09.300, 0, 2055, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "2026/12/03 01:50:19.000, 0, 900, 2070, 300.0, 0x0, Active, Not Active, Not Active, Not Active"]
    with open(c.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    t0 = time.mktime(time.strptime("2026/12/03 01:50:09", "%Y/%m/%d %H:%M:%S"))
    c.mark(t0, t0 + 1.0)
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2062.5 and s["reasons"] == ["sw_power_cap"]
    c.mark(t0 + 5.0, t0 + 6.0)
    assert c.summary()["samples"] == 0


def test_prefill_bytes_of_the_other_workloads():
    # fp32 B1 H1 L256 d32: q, k, v, log alpha, out in fp32 (5 x 128 B per token) + the final state
    assert bench.prefill_bytes(synth.FP32_SMALL) == 256 * 640 + 32 * 32 * 4 == 167936
    # elu+1 normalised, B4 H8 L2048 d64, no gate, no state written: q, k, v, out in bf16
    assert bench.prefill_bytes(synth.ELU_NORM, final_state=False) == 32 * 2048 * (3 * 128 + 128) == 33554432
    # gated B8 H16 L4096 d128, zero initial state, final state written
    assert bench.prefill_bytes(synth.PREFILL) == 128 * (4096 * (3 * 256 + 512 + 256) + 128 * 128 * 4) == 813694976


def test_backward_bytes_and_chunk_flops():
    # 128 heads x 4096 tokens x (q, k, v, dout bf16 4 x 256 + log alpha 512 + dq, dk, dv 3 x 512
    # + dlog_alpha 512)
    assert bench.bwd_bytes(synth.BWD) == 128 * 4096 * (1024 + 512 + 1536 + 512)
    # per chunk: six products over a C x C operand (D twice, P, and the masked parts of dQ, dK, dV:
    # 2 C^2 d each) and five over the state (dS, dQ, dG, dK, dV: 2 C d^2 each)
    per_chunk = 6 * 2 * 64 * 64 * 128 + 5 * 2 * 64 * 128 * 128
    assert bench.bwd_chunk_flops(synth.BWD) == 128 * 64 * per_chunk


def test_delta_bytes_and_chunk_flops():
    # 128 heads x (4096 tokens x (q, k, v 768 + beta 4 + log alpha 512 + out 256) + final state 64 KB)
    assert bench.delta_bytes(synth.DELTA) == 128 * (4096 * 1540 + 128 * 128 * 4)
    assert bench.delta_chunk_flops(synth.DELTA) == 128 * 64 * (4 * 2 * 64 * 64 * 128 + 3 * 2 * 64 * 128 * 128)
