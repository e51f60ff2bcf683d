"""Pins for the CPU oracle: each check ties it to something other than its own formulas.

* values the pages print (worked causal example, output lengths, GELU(1));
* special cases that reduce to library routines (numpy correlate/matmul, torch
  float64 conv1d / group_norm / layer_norm / gelu);
* closed-form invariants (GroupNorm mean 0 and variance s2/(s2+eps), scale
  invariance, row-min bias differences) and brute-force enumeration.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng_inputs(seed, N, Ci, Co, T, k, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        x = rng.integers(-3, 4, size=(N, Ci, T)).astype(np.float32)
        w = rng.integers(-3, 4, size=(Co, Ci, k)).astype(np.float32)
        b = rng.integers(-3, 4, size=(Co,)).astype(np.float32)
    else:
        x = rng.standard_normal((N, Ci, T)).astype(np.float32)
        w = rng.uniform(-0.5, 0.5, (Co, Ci, k)).astype(np.float32)
        b = rng.uniform(-0.5, 0.5, (Co,)).astype(np.float32)
    return x, w, b


def _torch_conv(x, w, b, stride, pl, pr, d):
    xt = F.pad(torch.from_numpy(x).double(), (pl, pr))
    return F.conv1d(xt, torch.from_numpy(w).double(), None if b is None else torch.from_numpy(b).double(),
                    stride=stride, dilation=d).numpy()


# ------------------------------------------------------------------------------------------ T_out

def test_t_out_page_values():
    for c in _golden("t_out_cases.json")["cases"]:
        assert oracle.t_out(c["T"], c["k"], c["stride"], c["pad_left"], c["pad_right"], c["dilation"]) == c["T_out"]


def test_t_out_brute_force_window_count():
    # Count window start positions that fit inside the padded sequence by enumeration.
    for T in range(1, 13):
        for k in range(1, 5):
            for s in (1, 2, 3):
                for d in (1, 2, 3):
                    for pl in range(0, 4):
                        for pr in range(0, 3):
                            padded = T + pl + pr
                            # output t reads padded[t*s], ..., padded[t*s + (k-1)*d]
                            count = sum(1 for t in range(padded) if t * s + (k - 1) * d <= padded - 1)
                            assert oracle.t_out(T, k, s, pl, pr, d) == count, (T, k, s, d, pl, pr)


# ------------------------------------------------------------------------------------------ conv

def test_causal_worked_example_from_page():
    g = _golden("causal_k4_worked_example.json")
    x = np.array(g["x"], dtype=np.float32).reshape(1, 1, -1)
    w = np.array(g["w"], dtype=np.float32).reshape(1, 1, -1)
    p = oracle.params(1, 1, 1, x.shape[2], g["k"], 1, g["pad_left"], g["pad_right"], g["dilation"])
    y = oracle.conv1d(p, x, w, None)
    assert y.shape == (1, 1, len(g["expected"]))
    assert np.array_equal(y[0, 0], np.array(g["expected"], dtype=np.float64))


@pytest.mark.parametrize("s,d,pl,pr,k", [(1, 1, 1, 1, 3), (1, 1, 3, 0, 4), (2, 1, 2, 1, 3), (1, 2, 4, 4, 5),
                                         (3, 2, 0, 5, 2), (1, 1, 0, 0, 1), (2, 3, 6, 0, 4)])
def test_delta_kernel_reproduces_shifted_input(s, d, pl, pr, k):
    # w[co][ci][kk] = [co == ci][kk == k0]  =>  y[n, c, t] = x[n, c, t*s + k0*d - pl] (0 outside [0, T)).
    N, C, T = 2, 3, 17
    x = np.random.default_rng(1).standard_normal((N, C, T)).astype(np.float32)
    To = oracle.t_out(T, k, s, pl, pr, d)
    for k0 in range(k):
        w = np.zeros((C, C, k), dtype=np.float32)
        for c in range(C):
            w[c, c, k0] = 1.0
        y = oracle.conv1d(oracle.params(N, C, C, T, k, s, pl, pr, d), x, w, None)
        exp = np.zeros((N, C, To))
        for t in range(To):
            pos = t * s + k0 * d - pl
            if 0 <= pos < T:
                exp[:, :, t] = x[:, :, pos]
        assert np.array_equal(y, exp)


@pytest.mark.parametrize("s,d,pl,pr,k", [(1, 1, 1, 1, 3), (1, 2, 4, 4, 5), (2, 1, 3, 0, 4), (1, 3, 0, 2, 2)])
def test_conv_integer_inputs_match_numpy_correlate(s, d, pl, pr, k):
    # Integer inputs make every sum exact; per (co, ci) pair the conv is numpy's
    # correlate of the zero-padded row with the dilated kernel, sampled every s.
    N, Ci, Co, T = 2, 2, 2, 5
    x, w, b = _rng_inputs(3, N, Ci, Co, T, k, integer=True)
    y = oracle.conv1d(oracle.params(N, Ci, Co, T, k, s, pl, pr, d), x, w, b)
    To = oracle.t_out(T, k, s, pl, pr, d)
    exp = np.zeros((N, Co, To))
    for n in range(N):
        for co in range(Co):
            acc = np.zeros(T + pl + pr - d * (k - 1))
            for ci in range(Ci):
                dil = np.zeros(d * (k - 1) + 1)
                dil[::d] = w[co, ci].astype(np.float64)
                acc += np.correlate(np.pad(x[n, ci].astype(np.float64), (pl, pr)), dil, mode="valid")
            exp[n, co] = acc[::s][:To] + b[co]
    assert np.array_equal(y, exp)


@pytest.mark.parametrize("shape", [(2, 5, 7, 33, 3, 1, 1, 1, 1), (3, 8, 4, 64, 4, 1, 3, 0, 1), (1, 6, 5, 50, 5, 2, 4, 4, 2),
                                   (2, 3, 9, 31, 2, 3, 0, 2, 3), (1, 16, 32, 128, 3, 1, 1, 1, 1)])
def test_conv_matches_torch_float64(shape):
    N, Ci, Co, T, k, s, pl, pr, d = shape
    x, w, b = _rng_inputs(5, N, Ci, Co, T, k)
    y = oracle.conv1d(oracle.params(N, Ci, Co, T, k, s, pl, pr, d), x, w, b)
    ref = _torch_conv(x, w, b, s, pl, pr, d)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_linear_is_conv_with_T1_k1():
    # Linear(rows x K -> C_out) is the conv with T = 1, k = 1 and no padding.
    M, K, Co = 9, 20, 11
    rng = np.random.default_rng(7)
    X = rng.standard_normal((M, K)).astype(np.float32)
    W = rng.standard_normal((Co, K)).astype(np.float32)
    b = rng.standard_normal(Co).astype(np.float32)
    y = oracle.conv1d(oracle.params(M, K, Co, 1, 1), X.reshape(M, K, 1), W.reshape(Co, K, 1), b)
    ref = X.astype(np.float64) @ W.astype(np.float64).T + b
    np.testing.assert_allclose(y[:, :, 0], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------ GroupNorm

def test_group_norm_matches_torch_float64():
    rng = np.random.default_rng(11)
    for (N, C, L, G) in [(2, 8, 5, 2), (3, 32, 17, 4), (1, 12, 1, 3), (2, 16, 9, 16), (2, 6, 7, 1)]:
        inp = rng.standard_normal((N, C, L)) * 3 + 1
        ga = rng.standard_normal(C).astype(np.float32)
        be = rng.standard_normal(C).astype(np.float32)
        out = oracle.group_norm(inp, G, 1e-5, ga, be)
        ref = F.group_norm(torch.from_numpy(inp), G, torch.from_numpy(ga).double(), torch.from_numpy(be).double(),
                           eps=float(np.float32(1e-5))).numpy()
        np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-10)


def test_group_norm_invariants():
    rng = np.random.default_rng(12)
    N, C, L, G, eps = 3, 16, 40, 4, np.float32(1e-5)
    inp = rng.standard_normal((N, C, L)) * 2.5 - 0.7
    out = oracle.group_norm(inp, G, eps)
    cpg = C // G
    for n in range(N):
        for g in range(G):
            grp_in = inp[n, g * cpg:(g + 1) * cpg]
            grp = out[n, g * cpg:(g + 1) * cpg]
            s2 = grp_in.var()
            assert abs(grp.mean()) < 1e-12
            assert abs(grp.var() - s2 / (s2 + float(eps))) < 1e-12
    # Positive scaling of the pre-norm values leaves the output unchanged up to eps effects.
    out2 = oracle.group_norm(inp * 37.0, G, eps)
    assert np.max(np.abs(out2 - out)) < 1e-5
    # A shift that is uniform within every group cancels exactly (up to rounding).
    shift = np.repeat(rng.standard_normal((N, G, 1)), cpg, axis=1)
    out3 = oracle.group_norm(inp + shift, G, eps)
    assert np.max(np.abs(out3 - out)) < 1e-12
    # G == C is instance norm, G == 1 is layer norm over (C, L).
    inst = F.instance_norm(torch.from_numpy(inp), eps=float(eps)).numpy()
    np.testing.assert_allclose(oracle.group_norm(inp, C, eps), inst, rtol=1e-10, atol=1e-10)
    ln = F.layer_norm(torch.from_numpy(inp), (C, L), eps=float(eps)).numpy()
    np.testing.assert_allclose(oracle.group_norm(inp, 1, eps), ln, rtol=1e-10, atol=1e-10)


def test_group_norm_rejects_bad_groups():
    with pytest.raises(ValueError):
        oracle.group_norm(np.zeros((1, 6, 3)), 4, 1e-5)


# ------------------------------------------------------------------------------------------ channel LayerNorm

def test_channel_layer_norm_matches_torch_float64():
    rng = np.random.default_rng(13)
    N, C, L = 3, 24, 11
    inp = rng.standard_normal((N, C, L)) * 1.7 + 0.3
    ga = rng.standard_normal(C).astype(np.float32)
    be = rng.standard_normal(C).astype(np.float32)
    out = oracle.channel_layer_norm(inp, 1e-5, ga, be)
    ref = F.layer_norm(torch.from_numpy(inp).transpose(1, 2), (C,), torch.from_numpy(ga).double(),
                       torch.from_numpy(be).double(), eps=float(np.float32(1e-5))).transpose(1, 2).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-10)
    plain = oracle.channel_layer_norm(inp, 1e-5)
    assert np.max(np.abs(plain.mean(axis=1))) < 1e-12


def test_channel_layer_norm_single_channel_gives_beta():
    inp = np.random.default_rng(1).standard_normal((2, 1, 5))
    be = np.array([0.25], dtype=np.float32)
    out = oracle.channel_layer_norm(inp, 1e-5, np.array([3.0], dtype=np.float32), be)
    assert np.all(out == 0.25)


# ------------------------------------------------------------------------------------------ GELU

def test_gelu_page_value_and_identities():
    for c in _golden("gelu_values.json")["cases"]:
        assert abs(oracle.gelu_erf(np.array([c["x"]]))[0] - c["gelu"]) < c["abs_tol"]
    z = np.linspace(-6, 6, 1201)
    g = oracle.gelu_erf(z)
    assert oracle.gelu_erf(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(g - oracle.gelu_erf(-z), z, atol=1e-14)
    ref = F.gelu(torch.from_numpy(z), approximate="none").numpy()
    np.testing.assert_allclose(g, ref, rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------------------------------------ row-min

def test_rowmin_bias_brute_force():
    rng = np.random.default_rng(14)
    N, C, L = 4, 37, 3
    inp = rng.standard_normal((N, C, L))
    inp[1, 5, 0] = inp[1, 9, 0] = inp[1].min() - 1.0  # a tie: lowest index wins
    bias2 = rng.standard_normal(C).astype(np.float32)
    out, am = oracle.rowmin_bias(inp, bias2)
    assert am[1, 0] == 5
    for n in range(N):
        for l in range(L):
            assert am[n, l] == int(np.argmin(inp[n, :, l]))
            m = inp[n, :, l].min()
            np.testing.assert_array_equal(out[n, :, l], m + bias2.astype(np.float64))
            # differences between channels are the bias differences
            np.testing.assert_allclose(out[n, :, l] - out[n, 0, l], bias2.astype(np.float64) - float(bias2[0]),
                                       atol=1e-12)


# ------------------------------------------------------------------------------------------ whole pipeline

def _torch_pipeline(wl, inp):
    y = torch.from_numpy(_torch_conv(inp["x"], inp["w"], inp["b"], wl.stride, wl.pad_left, wl.pad_right,
                                     wl.dilation))
    ga = None if inp["gamma"] is None else torch.from_numpy(inp["gamma"]).double()
    be = None if inp["beta"] is None else torch.from_numpy(inp["beta"]).double()
    eps = float(np.float32(wl.eps))
    if wl.norm == synth.NORM_GROUP:
        y = F.group_norm(y, wl.groups, ga, be, eps=eps)
    elif wl.norm == synth.NORM_CHANNEL_LAYER:
        y = F.layer_norm(y.transpose(1, 2), (wl.C_out,), ga, be, eps=eps).transpose(1, 2)
    am = None
    if wl.post == synth.POST_GELU_ERF:
        y = F.gelu(y, approximate="none")
    elif wl.post == synth.POST_ROWMIN_BIAS:
        m, am = torch.min(y, dim=1, keepdim=True)
        y = m + torch.from_numpy(inp["bias2"]).double().view(1, -1, 1)
        am = am[:, 0, :].numpy()
    return y.numpy(), am


def _shrunk(wl):
    # Keep each workload's structure (k, dilation, padding, norm, post-op, group size) at a size the
    # pure loops finish quickly.
    if wl.name == synth.LINEAR_GN_ROWMIN.name:
        return wl.replace(N=8, C_in=64, C_out=256, groups=16)
    if wl.name == synth.CAUSAL_CONV.name:
        return wl.replace(N=2, C_in=16, C_out=16, T=64)
    if wl.name == synth.CONV_LN_GELU_BF16.name:
        return wl.replace(N=2, C_in=16, C_out=32, T=48)
    if wl.name == synth.CONV_GN.name:
        return wl.replace(N=2, C_in=16, C_out=64, T=96, groups=8)
    return wl


@pytest.mark.parametrize("wl", synth.WORKLOADS, ids=lambda w: w.name)
def test_pipeline_matches_torch_float64_composition(wl):
    wl = _shrunk(wl)
    inp = synth.make_inputs(wl, seed=0)
    y, am = oracle.conv1d_norm(oracle.params_of(wl), inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"],
                               inp["bias2"])
    ref, ref_am = _torch_pipeline(wl, inp)
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-9)
    if ref_am is not None:
        assert np.array_equal(am, ref_am)


def test_samples_entry_matches_full_pipeline():
    wl = _shrunk(synth.CONV_GN)
    inp = synth.make_inputs(wl, seed=0)
    p = oracle.params_of(wl)
    y, _ = oracle.conv1d_norm(p, inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"])
    ys, _ = oracle.conv1d_norm_samples(p, [1, 0], inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"])
    assert np.array_equal(ys[0], y[1]) and np.array_equal(ys[1], y[0])


def test_thread_count_does_not_change_results():
    wl = _shrunk(synth.CONV_GN)
    inp = synth.make_inputs(wl, seed=0)
    p = oracle.params_of(wl)
    y1, _ = oracle.conv1d_norm(p, inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"], nthreads=1)
    y4, _ = oracle.conv1d_norm(p, inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"], nthreads=4)
    assert np.array_equal(y1, y4)


def test_oracle_rejects_invalid_shapes():
    assert oracle.t_out(2, 5, 1, 0, 0, 1) == 0
    assert oracle.t_out(4, 0, 1, 0, 0, 1) == -1
    with pytest.raises(ValueError):
        oracle.conv1d_norm(oracle.params(1, 1, 6, 8, 3, norm=1, groups=4), np.zeros((1, 1, 8), np.float32),
                           np.zeros((6, 1, 3), np.float32))


# ------------------------------------------------------------------ [p4]'s LayerNorm(W) + AvgPool3d + GELU
def _torch_ln_pool_gelu(z, eps, sw, ga, be):
    t = torch.from_numpy(z).double() + float(np.float32(sw))
    W = z.shape[-1]
    t = F.layer_norm(t, (W,), None if ga is None else torch.from_numpy(ga).double(),
                     None if be is None else torch.from_numpy(be).double(), eps=float(np.float32(eps)))
    t = F.avg_pool3d(t, kernel_size=2)
    return F.gelu(t, approximate="none").numpy()


@pytest.mark.parametrize("shape,affine", [((2, 3, 4, 6, 64), True), ((1, 2, 5, 7, 10), True),
                                          ((2, 1, 2, 2, 128), False), ((1, 1, 3, 3, 3), True)])
def test_ln_avgpool3d_gelu_matches_torch_float64(shape, affine):
    # [p4]'s second operator against the library composition in float64: layer_norm over the last
    # dimension, avg_pool3d(kernel 2) (odd extents floor), exact GELU
    rng = np.random.default_rng(11)
    z = rng.normal(0.5, 2.0, size=shape).astype(np.float32)
    W = shape[-1]
    ga = rng.normal(1.0, 0.1, size=W).astype(np.float32) if affine else None
    be = rng.normal(0.0, 0.1, size=W).astype(np.float32) if affine else None
    got = oracle.ln_avgpool3d_gelu(z, 1e-5, 1.0, ga, be)
    ref = _torch_ln_pool_gelu(z, 1e-5, 1.0, ga, be)
    assert got.shape == ref.shape
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_ln_avgpool3d_gelu_closed_forms():
    # rows constant along W: LayerNorm gives beta exactly, so every output is GELU of the mean of
    # beta over its two columns
    D, H, W = 4, 2, 8
    be = np.arange(W, dtype=np.float32) / 8.0
    z = np.broadcast_to(np.arange(D * H, dtype=np.float32).reshape(D, H, 1) * 3.0, (D, H, W)).copy()
    got = oracle.ln_avgpool3d_gelu(z[None], 1e-5, 0.0, None, be)[0]
    pair = (be[0::2].astype(np.float64) + be[1::2]) / 2.0
    expect = 0.5 * pair * (1.0 + np.array([math.erf(v / math.sqrt(2.0)) for v in pair]))
    for d2 in range(D // 2):
        for h2 in range(H // 2):
            np.testing.assert_allclose(got[d2, h2], expect, rtol=0, atol=1e-15)
    # a ramp along W: mean (W-1)/2, population variance (W^2-1)/12, so window w' averages to
    # (2w' + 1/2 - (W-1)/2) / sqrt(var + eps) whatever D and H
    W = 16
    ramp = np.broadcast_to(np.arange(W, dtype=np.float32), (2, 2, W)).copy()
    eps = np.float32(1e-5)
    got = oracle.ln_avgpool3d_gelu(ramp[None], float(eps), 0.0)[0][0, 0]
    var = (W * W - 1) / 12.0
    v = (2.0 * np.arange(W // 2) + 0.5 - (W - 1) / 2.0) / math.sqrt(var + float(eps))
    expect = 0.5 * v * (1.0 + np.array([math.erf(x / math.sqrt(2.0)) for x in v]))
    np.testing.assert_allclose(got, expect, rtol=0, atol=1e-14)


def test_ln_avgpool3d_gelu_sum_weight_cancels():
    # LayerNorm subtracts the row mean, so the scalar added before it cannot change the result
    rng = np.random.default_rng(5)
    z = rng.normal(size=(2, 4, 4, 32)).astype(np.float32)
    a = oracle.ln_avgpool3d_gelu(z, 1e-5, 0.0)
    b = oracle.ln_avgpool3d_gelu(z, 1e-5, 3.5)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ [p4]'s ConvTranspose3d
@pytest.mark.parametrize("shape", [(2, 3, 4, 3, 5, 4, 3, 2, 1, 1), (1, 2, 3, 3, 3, 2, 3, 1, 1, 0),
                                   (1, 4, 2, 2, 4, 3, 2, 2, 0, 1), (2, 2, 3, 2, 2, 5, 3, 3, 1, 2)])
def test_conv_transpose3d_matches_torch_float64(shape):
    # the gather form of the definition against the library's transposed convolution in float64
    N, Ci, Co, D, H, W, k, s, p, op = shape
    rng = np.random.default_rng(17)
    x = rng.normal(size=(N, Ci, D, H, W)).astype(np.float32)
    w = rng.uniform(-0.3, 0.3, size=(Ci, Co, k, k, k)).astype(np.float32)
    b = rng.uniform(-0.3, 0.3, size=Co).astype(np.float32)
    got = oracle.conv_transpose3d(x, w, b, stride=s, pad=p, out_pad=op)
    ref = F.conv_transpose3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(), torch.from_numpy(b).double(),
                             stride=s, padding=p, output_padding=op).numpy()
    assert got.shape == ref.shape
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_conv_transpose3d_scatter_form_and_page_shape():
    # the scatter form (every input voxel adds w * x at o = i*stride - pad + k, cropped), written
    # independently of the gather loops, on integers so both are exact; and the page's shape
    # arithmetic: x [.., 16, 32, 32], k 3, stride 2, pad 1, output pad 1 -> [.., 32, 64, 64]
    assert oracle.conv_transpose3d_shape(16, 32, 32, 3, 2, 1, 1) == (32, 64, 64)
    rng = np.random.default_rng(3)
    N, Ci, Co, D, H, W, k, s, p, op = 1, 2, 3, 3, 2, 4, 3, 2, 1, 1
    x = rng.integers(-3, 4, size=(N, Ci, D, H, W)).astype(np.float32)
    w = rng.integers(-2, 3, size=(Ci, Co, k, k, k)).astype(np.float32)
    Do, Ho, Wo = oracle.conv_transpose3d_shape(D, H, W, k, s, p, op)
    full = np.zeros((N, Co, (D - 1) * s + k + op, (H - 1) * s + k + op, (W - 1) * s + k + op))
    for n in range(N):
        for ci in range(Ci):
            for i in range(D):
                for j in range(H):
                    for l in range(W):
                        full[n, :, i * s:i * s + k, j * s:j * s + k, l * s:l * s + k] += x[n, ci, i, j, l] * w[ci]
    ref = full[:, :, p:p + Do, p:p + Ho, p:p + Wo]
    got = oracle.conv_transpose3d(x, w, None, stride=s, pad=p, out_pad=op)
    np.testing.assert_array_equal(got, ref)


def test_p4_model_conv_bias_cancels_in_layernorm():
    # The conv bias is one constant per channel, i.e. per LayerNorm row along W, so the page's model
    # (ConvTranspose3d, + scalar, LayerNorm over W, AvgPool3d, GELU) does not depend on it: the
    # one-pass kernel relies on this and normalizes the bare accumulators. (Tolerance: the float32
    # rounding of y + b, which the LayerNorm input goes through.)
    rng = np.random.default_rng(11)
    x = rng.normal(size=(1, 3, 2, 2, 4)).astype(np.float32)
    w = rng.uniform(-0.3, 0.3, size=(3, 4, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-2.0, 2.0, size=4).astype(np.float32)
    ga = rng.normal(1.0, 0.1, size=8).astype(np.float32)
    be = rng.normal(0.0, 0.1, size=8).astype(np.float32)
    with_b = oracle.conv_transpose3d(x, w, b, stride=2, pad=1, out_pad=1)[0].astype(np.float32)
    without = oracle.conv_transpose3d(x, w, None, stride=2, pad=1, out_pad=1)[0].astype(np.float32)
    assert not np.allclose(with_b, without)
    a1 = oracle.ln_avgpool3d_gelu(with_b, 1e-5, 1.0, ga, be)
    a0 = oracle.ln_avgpool3d_gelu(without, 1e-5, 0.0, ga, be)
    np.testing.assert_allclose(a1, a0, rtol=0, atol=2e-5)
