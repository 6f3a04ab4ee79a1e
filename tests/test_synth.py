"""Seeded input generator: determinism, index-addressed sampling, rounding."""
import numpy as np

import synth


def test_normals_are_deterministic_and_index_addressed():
    a = synth.normals(7, synth.T_Q, (1000,))
    b = synth.normals(7, synth.T_Q, (1000,))
    assert np.array_equal(a, b)
    c = synth.normals(7, synth.T_Q, (300,), start=500)
    assert np.array_equal(a[500:800], c)
    d = synth.normals(7, synth.T_K, (1000,))
    assert not np.array_equal(a, d)


def test_normals_moments():
    x = synth.normals(11, synth.T_V, (1 << 20,))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_large_threaded_generation_matches_serial():
    n = (1 << 22) + 12345
    x = synth.normals(3, synth.T_G, (n,))
    y = synth.normals(3, synth.T_G, (1000,), start=n - 1000)
    assert np.array_equal(x[-1000:], y)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is exactly halfway between bf16 1.0 and 1 + 2^-7: ties to even -> 1.0
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 0.0], dtype=np.float32)
    b = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f64(b)
    assert back[0] == 1.0 and back[1] == 1.0 + 2.0 ** -6 and back[2] == -2.5 and back[3] == 0.0


def test_head_sampling_matches_full_tensors():
    w = synth.with_shape(synth.LONGCTX, B=1, H=4, L=96, init_std=0.1)
    full = synth.make_prefill(w)
    part = synth.make_prefill(w, heads=[1, 3])
    for name in ("q", "k", "v", "log_alpha"):
        f = full[name].reshape(4, 96, -1)
        assert np.array_equal(part[name], f[[1, 3]])
    assert np.array_equal(part["init_state"], full["init_state"].reshape(4, 128, 256)[[1, 3]])


def test_log_alpha_recipe_range():
    w = synth.with_shape(synth.PREFILL, B=1, H=2, L=256)
    x = synth.make_prefill(w)
    la = x["log_alpha"]
    assert la.dtype == np.float32 and np.all(la < 0) and np.all(la > -1.0)


def test_decode_token_sampling():
    full = synth.decode_token(4, 3, 8, 8, step=5, seed=1)
    part = synth.decode_token(4, 3, 8, 8, step=5, seed=1, heads=[2, 7])
    assert np.array_equal(part["q"], full["q"].reshape(12, 8)[[2, 7]])
    assert np.array_equal(part["log_alpha"], full["log_alpha"].reshape(12, 8)[[2, 7]])
