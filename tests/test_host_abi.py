"""Host-only checks of the C ABI: the library loads, exports every declared symbol, validates
parameters and plans each workload; no device call is made."""
import ctypes
import os
import re

import pytest

import gemm_groupnorm_accelerator_gb300 as c1n
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "conv1d_norm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^(?:c1n_status|void|const char\*|int32_t)\s+(\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol():
    lib = c1n.load()
    declared = _declared_functions()
    assert set(declared) == set(c1n.EXPORTED_SYMBOLS), declared
    for name in declared:
        assert hasattr(lib, name), name
    assert c1n.conv1d_norm_version() >= 100


def _params(wl, **kw):
    d = dict(N=wl.N, C_in=wl.C_in, C_out=wl.C_out, T=wl.T, k=wl.k, stride=wl.stride, pad_left=wl.pad_left,
             pad_right=wl.pad_right, dilation=wl.dilation, norm=wl.norm, groups=wl.groups, eps=wl.eps, post=wl.post,
             dtype=wl.dtype)
    d.update(kw)
    return c1n.make_params(**d)


EXPECTED_PATH = {
    synth.CONV_GN_TINY.name: "tc_fused_gn",
    synth.CONV_GN.name: "tc_fused_gn",
    synth.CAUSAL_CONV.name: "tc_direct",
    synth.LINEAR_GN_ROWMIN.name: "tc_linear",
    synth.CONV_LN_GELU_BF16.name: "tc_fused_ln",
}


@pytest.mark.parametrize("wl", synth.WORKLOADS, ids=lambda w: w.name)
def test_plan_of_each_workload(wl):
    d = c1n.conv1d_norm_desc_create(_params(wl))
    try:
        info = c1n.conv1d_norm_plan_info(d)
        assert info.T_out == wl.T_out
        assert c1n.PATH_NAMES[info.path] == EXPECTED_PATH[wl.name]
        assert c1n.conv1d_norm_workspace_size(d) >= 256
        if info.path != c1n.PATH_SIMT:
            assert 16 <= info.mma_n <= 256 and info.mma_n % 16 == 0
            assert info.tile_t >= 1
    finally:
        c1n.conv1d_norm_destroy(d)


def test_conv_gn_cluster_geometry():
    d = c1n.conv1d_norm_desc_create(_params(synth.CONV_GN))
    info = c1n.conv1d_norm_plan_info(d)
    # 1024 steps in 8 tiles of 128; all 256 channels in one MMA N; one cluster of 8 CTAs per sample
    assert (info.cluster, info.tile_t, info.mma_n, info.n_tiles) == (8, 128, 256, 8 * 16)
    c1n.conv1d_norm_destroy(d)


@pytest.mark.parametrize("wl", [synth.CAUSAL_CONV, synth.LINEAR_GN_ROWMIN, synth.CONV_LN_GELU_BF16],
                         ids=lambda w: w.name)
def test_cta_pair_mainloop(wl):
    # CTA pairs: 256-row tiles, each CTA stages half of the B tile. AUTO pairs the Linear GEMM and
    # convolutions with at least 152 units of 256 rows; the 512-channel LayerNorm plan exchanges
    # statistics between single CTAs and does not pair.
    paired = wl is not synth.CONV_LN_GELU_BF16
    d = c1n.conv1d_norm_desc_create(_params(wl))
    info = c1n.conv1d_norm_plan_info(d)
    assert (info.cta_pair, info.tile_t) == ((1, 256) if paired else (0, 128))
    c1n.conv1d_norm_destroy(d)
    # a small convolution keeps one CTA per 128-row tile under AUTO; SINGLE and PAIR force either
    small = synth.CAUSAL_CONV.replace(N=2, T=1024)
    for mainloop, want in ((c1n.MAINLOOP_AUTO, 0), (c1n.MAINLOOP_SINGLE, 0), (c1n.MAINLOOP_PAIR, 1)):
        d = c1n.conv1d_norm_desc_create(_params(small, mainloop=mainloop))
        assert c1n.conv1d_norm_plan_info(d).cta_pair == want
        c1n.conv1d_norm_destroy(d)
    d = c1n.conv1d_norm_desc_create(_params(synth.CAUSAL_CONV, mainloop=c1n.MAINLOOP_SINGLE))
    assert c1n.conv1d_norm_plan_info(d).cta_pair == 0
    c1n.conv1d_norm_destroy(d)
    # (the 512-channel LayerNorm cluster plan exchanges statistics between single CTAs: pairs need
    # the two-pass plan there)
    forced = c1n.PATH_TC_TWO_PASS if wl is synth.CONV_LN_GELU_BF16 else -1
    d = c1n.conv1d_norm_desc_create(_params(wl, mainloop=c1n.MAINLOOP_PAIR, force_path=forced))
    info = c1n.conv1d_norm_plan_info(d)
    assert (info.cta_pair, info.tile_t, info.mma_n) == (1, 256, 256)
    c1n.conv1d_norm_destroy(d)
    if wl is synth.CONV_LN_GELU_BF16:
        with pytest.raises(c1n.C1NError) as e:
            c1n.conv1d_norm_desc_create(_params(wl, mainloop=c1n.MAINLOOP_PAIR))
        assert e.value.status == c1n.ERR_UNSUPPORTED
    d = c1n.conv1d_norm_desc_create(_params(wl, mainloop=c1n.MAINLOOP_SINGLE))
    info = c1n.conv1d_norm_plan_info(d)
    assert (info.cta_pair, info.tile_t) == (0, 128)
    c1n.conv1d_norm_destroy(d)


def test_layer_norm_cluster_plan():
    # 512 channels: two CTAs per 128-step tile (a cluster of two), 256 channels and two accumulators each
    d = c1n.conv1d_norm_desc_create(_params(synth.CONV_LN_GELU_BF16))
    info = c1n.conv1d_norm_plan_info(d)
    assert (c1n.PATH_NAMES[info.path], info.cluster, info.mma_n, info.tile_t) == ("tc_fused_ln", 2, 256, 128)
    assert info.n_tiles == synth.CONV_LN_GELU_BF16.N * synth.CONV_LN_GELU_BF16.T_out // 128
    c1n.conv1d_norm_destroy(d)
    d = c1n.conv1d_norm_desc_create(_params(synth.CONV_LN_GELU_BF16, C_out=256))
    assert c1n.conv1d_norm_plan_info(d).cluster == 1
    c1n.conv1d_norm_destroy(d)


def test_cta_pair_refused_where_the_plan_cannot_pair():
    # fused GroupNorm exchanges statistics between single CTAs; MMA N = 48 does not split in two 16-row halves
    for wl in (synth.CONV_GN, synth.CAUSAL_CONV.replace(C_out=48)):
        with pytest.raises(c1n.C1NError) as e:
            c1n.conv1d_norm_desc_create(_params(wl, mainloop=c1n.MAINLOOP_PAIR))
        assert e.value.status == c1n.ERR_UNSUPPORTED
    d = c1n.conv1d_norm_desc_create(_params(synth.CONV_GN))
    assert c1n.conv1d_norm_plan_info(d).cta_pair == 0
    c1n.conv1d_norm_destroy(d)


def test_tensor_x3_plans():
    # 3xTF32: fp32 convolution plans only; the packed weights hold the TF32 head and tail
    base = c1n.conv1d_norm_desc_create(_params(synth.CONV_GN))
    d = c1n.conv1d_norm_desc_create(_params(synth.CONV_GN, math=c1n.MATH_TENSOR_X3))
    assert c1n.PATH_NAMES[c1n.conv1d_norm_plan_info(d).path] == "tc_fused_gn"
    assert c1n.conv1d_norm_workspace_size(d) > c1n.conv1d_norm_workspace_size(base)
    c1n.conv1d_norm_destroy(d)
    c1n.conv1d_norm_destroy(base)
    for wl in (synth.CONV_LN_GELU_BF16, synth.LINEAR_GN_ROWMIN):
        with pytest.raises(c1n.C1NError) as e:
            c1n.conv1d_norm_desc_create(_params(wl, math=c1n.MATH_TENSOR_X3))
        assert e.value.status == c1n.ERR_UNSUPPORTED


def test_simt_forced_and_tensor_forced():
    wl = synth.CONV_GN_TINY
    d = c1n.conv1d_norm_desc_create(_params(wl, math=c1n.MATH_SIMT))
    assert c1n.conv1d_norm_plan_info(d).path == c1n.PATH_SIMT
    c1n.conv1d_norm_destroy(d)
    # No silent fallback: shapes without a tensor-core plan (stride 2; T not a multiple of 16 bytes
    # of elements) are refused under AUTO as under TENSOR, and run on the SIMT path only when the
    # caller asks for it.
    for bad in (dict(stride=2), dict(T=77), dict(T=126)):
        for math in (c1n.MATH_AUTO, c1n.MATH_TENSOR):
            with pytest.raises(c1n.C1NError) as e:
                c1n.conv1d_norm_desc_create(_params(wl, math=math, **bad))
            assert e.value.status == c1n.ERR_UNSUPPORTED
            assert "SIMT" in str(e.value) or math == c1n.MATH_TENSOR
        d = c1n.conv1d_norm_desc_create(_params(wl, math=c1n.MATH_SIMT, **bad))
        assert c1n.conv1d_norm_plan_info(d).path == c1n.PATH_SIMT
        c1n.conv1d_norm_destroy(d)
    d = c1n.conv1d_norm_desc_create(_params(wl, force_path=c1n.PATH_TC_TWO_PASS))
    assert c1n.conv1d_norm_plan_info(d).path == c1n.PATH_TC_TWO_PASS
    c1n.conv1d_norm_destroy(d)


def test_halo_past_one_staged_box_is_refused():
    # (k - 1) d = 120 rows is the longest halo a staged x box (256 time steps) holds with the tile's
    # 128 rows; one more dilation step is refused by the tensor-core plans (SIMT still takes it)
    wl = synth.CAUSAL_CONV.replace(N=2, C_in=32, C_out=64, T=512, k=16, dilation=8, pad_left=120, pad_right=0)
    d = c1n.conv1d_norm_desc_create(_params(wl))
    assert c1n.PATH_NAMES[c1n.conv1d_norm_plan_info(d).path] == "tc_direct"
    c1n.conv1d_norm_destroy(d)
    far = wl.replace(dilation=9, pad_left=135)
    with pytest.raises(c1n.C1NError) as e:
        c1n.conv1d_norm_desc_create(_params(far))
    assert e.value.status == c1n.ERR_UNSUPPORTED
    d = c1n.conv1d_norm_desc_create(_params(far, math=c1n.MATH_SIMT))
    assert c1n.conv1d_norm_plan_info(d).path == c1n.PATH_SIMT
    c1n.conv1d_norm_destroy(d)
    with pytest.raises(c1n.C1NError) as e:  # more than 16 taps
        c1n.conv1d_norm_desc_create(_params(wl.replace(k=17, dilation=1, pad_left=16)))
    assert e.value.status == c1n.ERR_UNSUPPORTED


@pytest.mark.parametrize("bad", [dict(N=0), dict(C_in=0), dict(k=0), dict(stride=0), dict(dilation=0),
                                 dict(pad_left=-1), dict(groups=3), dict(eps=0.0), dict(eps=float("nan")),
                                 dict(norm=7), dict(post=5), dict(dtype=3), dict(math=9), dict(math=4), dict(T=2, k=5),
                                 dict(force_path=11), dict(mainloop=3), dict(mainloop=-1)])
def test_invalid_params_are_rejected(bad):
    with pytest.raises(c1n.C1NError) as e:
        c1n.conv1d_norm_desc_create(_params(synth.CONV_GN_TINY, **bad))
    assert e.value.status == c1n.ERR_INVALID_ARG
    assert c1n.load().conv1d_norm_last_error()


def test_run_without_workspace_and_null_pointers():
    d = c1n.conv1d_norm_desc_create(_params(synth.CONV_GN_TINY))
    lib = c1n.load()
    # no workspace attached
    st = lib.conv1d_norm_run(d, 16, 16, None, None, None, 16, None)
    assert st == c1n.ERR_WORKSPACE
    assert c1n.conv1d_norm_set_workspace(d, 0, 0) is None
    with pytest.raises(c1n.C1NError) as e:
        c1n.conv1d_norm_set_workspace(d, 256, 16)
    assert e.value.status == c1n.ERR_WORKSPACE
    with pytest.raises(c1n.C1NError) as e:
        c1n.conv1d_norm_set_workspace(d, 1024 + 8, 1 << 30)
    assert e.value.status == c1n.ERR_ALIGNMENT
    # NULL x is an argument error whatever the workspace
    args = c1n.Args(None, 16, None, None, None, None, 16, None, 4096, 1 << 30, 0)
    assert lib.conv1d_norm_run_ex(d, ctypes.byref(args), None) == c1n.ERR_INVALID_ARG
    c1n.conv1d_norm_destroy(d)


def test_rowmin_needs_run_ex_and_bias2():
    d = c1n.conv1d_norm_desc_create(_params(synth.LINEAR_GN_ROWMIN))
    lib = c1n.load()
    assert lib.conv1d_norm_run(d, 16, 16, None, None, None, 16, None) == c1n.ERR_INVALID_ARG
    args = c1n.Args(16, 16, None, None, None, None, 16, None, 4096, 1 << 40, 0)
    assert lib.conv1d_norm_run_ex(d, ctypes.byref(args), None) == c1n.ERR_INVALID_ARG
    c1n.conv1d_norm_destroy(d)


def test_profiling_toggle_without_a_run():
    d = c1n.conv1d_norm_desc_create(_params(synth.CONV_GN_TINY))
    c1n.conv1d_norm_set_profiling(d, True)
    assert c1n.conv1d_norm_kernel_times(d) == []  # no profiled run yet
    c1n.conv1d_norm_set_profiling(d, False)
    c1n.conv1d_norm_destroy(d)


def test_status_strings():
    for s in range(8):
        assert c1n.conv1d_norm_status_string(s)


def test_ln_avgpool3d_gelu_validation_without_device():
    # argument errors are reported before anything touches a device
    z = ctypes.c_void_p(4096)  # never dereferenced: every call below fails validation first
    ok = c1n.LnPoolParams(2, 3, 4, 4, 64, 1e-5)
    cases = [
        (c1n.LnPoolParams(0, 3, 4, 4, 64, 1e-5), z.value, z.value, c1n.ERR_INVALID_ARG),
        (c1n.LnPoolParams(2, 3, 4, 4, 64, 0.0), z.value, z.value, c1n.ERR_INVALID_ARG),
        (c1n.LnPoolParams(2, 3, 4, 4, 48, 1e-5), z.value, z.value, c1n.ERR_UNSUPPORTED),
        (c1n.LnPoolParams(2, 3, 4, 4, 96, 1e-5), z.value, z.value, c1n.ERR_UNSUPPORTED),
        (ok, None, z.value, c1n.ERR_INVALID_ARG),
        (ok, z.value + 4, z.value, c1n.ERR_ALIGNMENT),
        (ok, z.value, z.value + 8, c1n.ERR_ALIGNMENT),
    ]
    for p, zp, op, status in cases:
        with pytest.raises(c1n.C1NError) as e:
            c1n.ln_avgpool3d_gelu_run(p, zp, 1.0, None, None, op, 0)
        assert e.value.status == status, (p.W, p.eps, status)
    # no pooling window (D or H below 2): nothing to do, nothing launched
    c1n.ln_avgpool3d_gelu_run(c1n.LnPoolParams(2, 3, 1, 4, 64, 1e-5), z.value, 1.0, None, None, z.value, 0)


def test_conv_transpose3d_validation_without_device():
    p = lambda **kw: c1n.ConvT3dParams(*[kw.get(k, v) for k, v in (("N", 2), ("C_in", 4), ("C_out", 64), ("D", 3),
                                                                   ("H", 3), ("W", 3), ("k", 3), ("stride", 2),
                                                                   ("pad", 1), ("out_pad", 1), ("math", 0))])
    x = ctypes.c_void_p(4096).value
    for params, status in ((p(N=0), c1n.ERR_INVALID_ARG), (p(k=5), c1n.ERR_UNSUPPORTED), (p(stride=1), c1n.ERR_UNSUPPORTED),
                           (p(pad=0), c1n.ERR_UNSUPPORTED), (p(out_pad=2), c1n.ERR_UNSUPPORTED),
                           (p(C_out=48), c1n.ERR_UNSUPPORTED)):
        with pytest.raises(c1n.C1NError) as e:
            c1n.conv_transpose3d_run(params, x, x, None, x, None, 0, 0)
        assert e.value.status == status
    with pytest.raises(c1n.C1NError) as e:
        c1n.conv_transpose3d_run(p(), None, x, None, x, None, 0, 0)
    assert e.value.status == c1n.ERR_INVALID_ARG
    # plan choice: the tensor cores take C_in 32 / C_out 64 (and need a workspace), else CUDA cores
    assert c1n.conv_transpose3d_workspace_size(p(C_in=32, W=32)) > 0
    assert c1n.conv_transpose3d_workspace_size(p(C_in=16)) == 0
    assert c1n.conv_transpose3d_workspace_size(p(C_in=32, W=32, math=1)) == 0
    with pytest.raises(c1n.C1NError) as e:
        c1n.conv_transpose3d_workspace_size(p(C_in=16, math=2))
    assert e.value.status == c1n.ERR_UNSUPPORTED
    with pytest.raises(c1n.C1NError) as e:  # the tensor-core plan without its workspace
        c1n.conv_transpose3d_run(p(C_in=32, W=32), x, x, None, x, None, 0, 0)
    assert e.value.status == c1n.ERR_WORKSPACE


def test_fused_p4_model_validation_without_device():
    # the one-pass model takes the page's shape only (C_in 32, C_out 64, W 32, k 3, stride 2, pad 1,
    # output pad 1); everything is checked before any device call
    p = lambda **kw: c1n.ConvT3dParams(*[kw.get(k, v) for k, v in (("N", 2), ("C_in", 32), ("C_out", 64), ("D", 3),
                                                                   ("H", 5), ("W", 32), ("k", 3), ("stride", 2),
                                                                   ("pad", 1), ("out_pad", 1), ("math", 0))])
    x = ctypes.c_void_p(4096).value
    need = c1n.conv_transpose3d_ln_avgpool3d_gelu_workspace_size(p())
    # status word + channels-last x + two channel halves of 864 packed weight rows
    assert need == 256 + (2 * 32 * 3 * 5 * 32 * 4 + 1023) // 1024 * 1024 + 2 * 864 * 128
    for params, status in ((p(N=0), c1n.ERR_INVALID_ARG), (p(W=16), c1n.ERR_UNSUPPORTED),
                           (p(C_in=16), c1n.ERR_UNSUPPORTED), (p(C_out=32), c1n.ERR_UNSUPPORTED),
                           (p(out_pad=0), c1n.ERR_UNSUPPORTED), (p(k=5), c1n.ERR_UNSUPPORTED)):
        with pytest.raises(c1n.C1NError) as e:
            c1n.conv_transpose3d_ln_avgpool3d_gelu_run(params, 1e-5, 1.0, x, x, None, None, None, x, x, need, 0)
        assert e.value.status == status
    bad = ((dict(eps=0.0), c1n.ERR_INVALID_ARG), (dict(x=None), c1n.ERR_INVALID_ARG),
           (dict(ws_bytes=need - 1), c1n.ERR_WORKSPACE), (dict(ws=x + 16), c1n.ERR_ALIGNMENT),
           (dict(out=x + 4), c1n.ERR_ALIGNMENT))
    for kw, status in bad:
        a = dict(eps=1e-5, x=x, out=x, ws=x, ws_bytes=need)
        a.update(kw)
        with pytest.raises(c1n.C1NError) as e:
            c1n.conv_transpose3d_ln_avgpool3d_gelu_run(p(), a["eps"], 1.0, a["x"], x, None, None, None, a["out"], a["ws"],
                                                       a["ws_bytes"], 0)
        assert e.value.status == status


def test_static_scratch_refuses_prepacked_weights_without_device():
    # The entry point without allocation shares one array among all descriptors, so weights packed
    # by an earlier call may be another operator's: it refuses the flag before touching the device.
    d = c1n.conv1d_norm_desc_create(_params(synth.CONV_GN_TINY))
    lib = c1n.load()
    args = c1n.Args(16, 16, None, None, None, None, 16, None, None, 0, c1n.FLAG_WEIGHTS_PACKED)
    assert lib.conv1d_norm_run_static_scratch(d, ctypes.byref(args), None) == c1n.ERR_INVALID_ARG
    assert b"WEIGHTS_PACKED" in lib.conv1d_norm_last_error()
    args = c1n.Args(16, 16, None, None, None, None, 16, None, 4096, 1 << 20, 0)  # a workspace is refused too
    assert lib.conv1d_norm_run_static_scratch(d, ctypes.byref(args), None) == c1n.ERR_INVALID_ARG
    c1n.conv1d_norm_destroy(d)
