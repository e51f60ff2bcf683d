"""The seeded input generator: determinism, prefix stability and the stated distributions."""
import numpy as np

import synth


def test_generator_is_deterministic_and_streams_differ():
    a = synth.normal(0, synth.STREAM_X, 1000)
    b = synth.normal(0, synth.STREAM_X, 1000)
    c = synth.normal(0, synth.STREAM_W, 1000)
    d = synth.normal(1, synth.STREAM_X, 1000)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_prefix_is_stable():
    full = synth.normal(0, synth.STREAM_X, 10000)
    assert np.array_equal(full[:1234], synth.normal(0, synth.STREAM_X, 1234))
    wl = synth.CONV_GN_TINY
    x_full = synth.make_inputs(wl)["x"]
    x_one = synth.make_inputs(wl, n_rows=1)["x"]
    assert np.array_equal(x_full[:1], x_one)


def test_distributions():
    z = synth.normal(0, synth.STREAM_X, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    u = synth.uniform_pm(0, synth.STREAM_W, 400000, 0.25)
    assert u.min() >= -0.25 and u.max() <= 0.25
    assert abs(u.std() - 0.25 / np.sqrt(3)) < 1e-3
    g = synth.normal(0, synth.STREAM_GAMMA, 400000, 1.0, 0.1)
    assert abs(g.mean() - 1.0) < 1e-3 and abs(g.std() - 0.1) < 1e-3


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e-3], dtype=np.float32)
    r = synth.round_bf16(vals)
    # ties go to the even mantissa: 1 + 2^-8 -> 1.0, 1 + 3*2^-8 -> 1 + 2^-6
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == np.float32(1.0 + 2 ** -6)
    bits = r.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)
    assert np.all(np.abs(r - vals) <= np.abs(vals) * 2 ** -8)


def test_workload_shapes():
    assert synth.CONV_GN.T_out == 1024 and synth.CAUSAL_CONV.T_out == 8192
    assert synth.CONV_LN_GELU_BF16.T_out == 4096 and synth.LINEAR_GN_ROWMIN.T_out == 1
    assert synth.CONV_GN.gemm_mnk == (16384, 256, 384)
    assert synth.CAUSAL_CONV.gemm_mnk == (262144, 256, 1024)
    assert synth.LINEAR_GN_ROWMIN.gemm_mnk == (1024, 8192, 8192)
    assert synth.CONV_LN_GELU_BF16.gemm_mnk == (262144, 512, 1280)
