"""GPU parity: the CUDA library, called through the C ABI, against the CPU oracle on the same seeded
inputs. Tolerances (max abs error): 1e-4 for the SIMT fp32 path, 5e-3 for the TF32 tensor-core
path, 3e-2 for bf16 data; row-min argmin must agree wherever the minimum is unique by > 1e-2."""
import functools

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_SIMT, TOL_TF32, TOL_BF16 = 1e-4, 5e-3, 3e-2


def _tol(wl, path):
    if wl.dtype == synth.DTYPE_BF16:
        return TOL_BF16
    return TOL_SIMT if path == "simt" else TOL_TF32


@functools.lru_cache(maxsize=8)
def _inputs(wl):
    return synth.make_inputs(wl, seed=0)


def _to_dev(a, bf16):
    if a is None:
        return None
    t = torch.from_numpy(a).cuda()
    return t.to(torch.bfloat16) if bf16 else t


def run_gpu(c1n, wl, inp, math=0, force_path=-1, mainloop=0):
    params = c1n.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation,
                             wl.norm, wl.groups, wl.eps, wl.post, wl.dtype, math, force_path, mainloop)
    op = c1n.Conv1dNorm(params)
    bf = wl.dtype == synth.DTYPE_BF16
    x, w = _to_dev(inp["x"], bf), _to_dev(inp["w"], bf)
    b, ga, be, b2 = (_to_dev(inp[k], False) for k in ("b", "gamma", "beta", "bias2"))
    out = torch.full((wl.N, wl.C_out, op.T_out), float("nan"), dtype=op.out_dtype(), device="cuda")
    am = torch.full((wl.N, op.T_out), -1, dtype=torch.int32, device="cuda") if wl.post == synth.POST_ROWMIN_BIAS else None
    op(x, w, b, ga, be, bias2=b2, out=out, argmin=am)
    torch.cuda.synchronize()
    op.check()
    path = op.path
    y = out.float().cpu().numpy()
    return y, (None if am is None else am.cpu().numpy()), path


def compare(wl, y, am, ref, ref_am, path, label="", tol=None):
    assert np.all(np.isfinite(y)), f"{label}: non-finite output (unwritten elements?)"
    err = float(np.max(np.abs(y.astype(np.float64) - ref)))
    tol = _tol(wl, path) if tol is None else tol
    assert err <= tol, f"{label} path={path}: max abs err {err:.3e} > {tol}"
    if ref_am is not None:
        # argmin must match where the minimum is unique by a margin > 1e-2
        assert am is not None
        # recompute margins from the oracle's pre-broadcast values: y - bias2 is the row minimum,
        # so margins need the normalized values; the caller passes them through `ref_margin`.
    return err


def oracle_full(wl, inp):
    return oracle.conv1d_norm(oracle.params_of(wl), inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"],
                              inp["bias2"])


def _argmin_margin(wl, inp, ns=None):
    """Oracle normalized values before the row-min, to find rows whose minimum is unique by > 1e-2."""
    pre = wl.replace(post=synth.POST_NONE)
    if ns is None:
        z, _ = oracle_full(pre, inp)
    else:
        z, _ = oracle.conv1d_norm_samples(oracle.params_of(pre), ns, inp["x"], inp["w"], inp["b"], inp["gamma"],
                                          inp["beta"])
    s = np.sort(z, axis=1)
    return s[:, 1, :] - s[:, 0, :]


def check_argmin(am, ref_am, margin):
    sel = margin > 1e-2
    assert sel.any()
    assert np.array_equal(am[sel], ref_am[sel]), f"argmin mismatch on {(am[sel] != ref_am[sel]).sum()} rows"


# ------------------------------------------------------------------------------ small shapes, every path

SMALL = {
    "gn_tiny": synth.CONV_GN_TINY,
    "gn_c2_structure": synth.CONV_GN.replace(N=3, C_in=40, C_out=200, T=1000, groups=25),
    "gn_cpg1": synth.CONV_GN.replace(N=2, C_in=32, C_out=64, T=256, groups=64),
    "gn_cpg128": synth.CONV_GN.replace(N=2, C_in=32, C_out=256, T=256, groups=2),
    "gn_cpg4": synth.CONV_GN.replace(N=2, C_in=32, C_out=64, T=384, groups=16),
    "gn_cpg16": synth.CONV_GN.replace(N=3, C_in=40, C_out=128, T=512, groups=8),
    "gn_cpg25": synth.CONV_GN.replace(N=2, C_in=16, C_out=200, T=256, groups=8),
    # T_out = 251: rows are not 16-byte multiples, so the fused tile is stored without TMA
    "gn_ragged_out": synth.CONV_GN.replace(N=2, C_in=24, C_out=48, T=252, k=4, groups=6),
    "gn_g1_twopass": synth.CONV_GN.replace(N=2, C_in=32, C_out=256, T=128, groups=1),
    "gn_gelu": synth.CONV_GN.replace(N=2, C_in=24, C_out=96, T=320, groups=12, post=synth.POST_GELU_ERF),
    "causal_k4": synth.CAUSAL_CONV.replace(N=2, C_in=64, C_out=160, T=1024),
    # enough 128-step tiles that each persistent CTA (one per SM) runs 2, then about 4 work units
    "causal_units2": synth.CAUSAL_CONV.replace(N=2, C_in=32, C_out=64, T=152 * 128),
    "causal_units4": synth.CAUSAL_CONV.replace(N=4, C_in=32, C_out=64, T=160 * 128),
    "conv_k1": synth.CAUSAL_CONV.replace(N=2, C_in=36, C_out=130, T=300, k=1, pad_left=0),
    "conv_dil3_pads": synth.CAUSAL_CONV.replace(N=2, C_in=20, C_out=64, T=412, k=3, pad_left=5, pad_right=2,
                                                dilation=3, w_bound=0.2),
    "conv_nopad": synth.CAUSAL_CONV.replace(N=3, C_in=16, C_out=48, T=96, k=5, pad_left=0, w_bound=0.2),
    "conv_gelu": synth.CAUSAL_CONV.replace(N=2, C_in=32, C_out=32, T=128, post=synth.POST_GELU_ERF),
    "conv_rowmin": synth.CAUSAL_CONV.replace(N=2, C_in=32, C_out=40, T=64, post=synth.POST_ROWMIN_BIAS),
    "linear_rowmin": synth.LINEAR_GN_ROWMIN.replace(N=200, C_in=72, C_out=320, groups=20),
    "linear_plain": synth.LINEAR_GN_ROWMIN.replace(N=130, C_in=64, C_out=96, norm=synth.NORM_NONE,
                                                   post=synth.POST_NONE),
    "linear_gn_gelu": synth.LINEAR_GN_ROWMIN.replace(N=150, C_in=96, C_out=512, groups=64, post=synth.POST_GELU_ERF),
    "linear_gn_cpg32_bf16": synth.LINEAR_GN_ROWMIN.replace(N=140, C_in=128, C_out=256, groups=8,
                                                           post=synth.POST_NONE, dtype=synth.DTYPE_BF16),
    "linear_rowmin_nonorm": synth.LINEAR_GN_ROWMIN.replace(N=70, C_in=64, C_out=288, norm=synth.NORM_NONE),
    "linear_gn_cpg4_twopass": synth.LINEAR_GN_ROWMIN.replace(N=66, C_in=32, C_out=96, groups=24),
    "linear_gelu_nonorm": synth.LINEAR_GN_ROWMIN.replace(N=140, C_in=48, C_out=96, norm=synth.NORM_NONE,
                                                         post=synth.POST_GELU_ERF),
    "ln_gelu_bf16": synth.CONV_LN_GELU_BF16.replace(N=2, C_in=48, C_out=160, T=264),
    "ln_c384_f32": synth.CONV_LN_GELU_BF16.replace(N=2, C_in=40, C_out=384, T=200, dtype=synth.DTYPE_F32,
                                                   post=synth.POST_NONE),
    "ln_c512_bf16": synth.CONV_LN_GELU_BF16.replace(N=2, C_in=64, C_out=512, T=320),
    "gn_bf16": synth.CONV_GN.replace(N=2, C_in=64, C_out=128, T=512, groups=16, dtype=synth.DTYPE_BF16),
    "conv_bf16": synth.CAUSAL_CONV.replace(N=2, C_in=72, C_out=136, T=400, dtype=synth.DTYPE_BF16),
    # two channel blocks of 192: 64-channel groups stay inside a block; 128-channel groups straddle
    "gn_cb2": synth.CONV_GN.replace(N=2, C_in=32, C_out=384, T=640, groups=6),
    "gn_cb2_straddle": synth.CONV_GN.replace(N=2, C_in=32, C_out=384, T=640, groups=3),
    # 16 tiles of 128 steps, the last one 80 steps long
    "gn_long_ragged": synth.CONV_GN.replace(N=2, C_in=32, C_out=64, T=2000, groups=8),
    # three channel blocks (224, 224, 192): channel LayerNorm takes the two-pass plan
    "ln_c640_f32": synth.CONV_LN_GELU_BF16.replace(N=2, C_in=40, C_out=640, T=200, dtype=synth.DTYPE_F32,
                                                   post=synth.POST_NONE),
    # the most taps (16) and the longest halo one staged x box holds ((k - 1) d = 120 rows)
    "conv_k16_maxhalo": synth.CAUSAL_CONV.replace(N=2, C_in=32, C_out=64, T=512, k=16, dilation=8, pad_left=120,
                                                  pad_right=0),
    "gn_k16_d2": synth.CONV_GN.replace(N=2, C_in=32, C_out=64, T=256, k=16, dilation=2, pad_left=15, pad_right=15,
                                       groups=8),
    "ln_bf16_k16_maxhalo": synth.CONV_LN_GELU_BF16.replace(N=2, C_in=64, C_out=128, T=256, k=16, dilation=8,
                                                           pad_left=56, pad_right=64),
    "stride2_simt": synth.CONV_GN.replace(N=2, C_in=16, C_out=32, T=101, stride=2, groups=8),
    "odd_T_simt": synth.CAUSAL_CONV.replace(N=2, C_in=8, C_out=24, T=77),
}
# shapes no tensor-core plan takes: refused unless the caller asks for the SIMT path
TC_REFUSED = {"stride2_simt", "odd_T_simt"}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("mode", ["auto", "simt", "single", "pair"])
def test_small_shapes(cuda_lib, name, mode):
    # auto: the planner's choice; single: one CTA per 128-row tile; pair: CTA-pair (cta_group::2)
    # mainloop where the plan allows it; simt: the fp32 CUDA-core check path
    wl = SMALL[name]
    math = 1 if mode == "simt" else 0
    mainloop = {"single": cuda_lib.MAINLOOP_SINGLE, "pair": cuda_lib.MAINLOOP_PAIR}.get(mode, cuda_lib.MAINLOOP_AUTO)
    if name in TC_REFUSED and math == 0:
        with pytest.raises(cuda_lib.C1NError) as e:
            cuda_lib.conv1d_norm_desc_create(cuda_lib.make_params(
                wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation, wl.norm,
                wl.groups, wl.eps, wl.post, wl.dtype, 0, -1, mainloop))
        assert e.value.status == cuda_lib.ERR_UNSUPPORTED
        return
    inp = _inputs(wl)
    ref, ref_am = oracle_full(wl, inp)
    if mode == "pair":
        try:
            cuda_lib.conv1d_norm_destroy(cuda_lib.conv1d_norm_desc_create(cuda_lib.make_params(
                wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation, wl.norm,
                wl.groups, wl.eps, wl.post, wl.dtype, 0, -1, mainloop)))
        except cuda_lib.C1NError:
            pytest.skip("plan cannot run on CTA pairs")
    y, am, path = run_gpu(cuda_lib, wl, inp, math=math, mainloop=mainloop)
    if math == 1:
        assert path == "simt"
    compare(wl, y, am, ref, ref_am, path, name)
    if ref_am is not None:
        check_argmin(am, ref_am, _argmin_margin(wl, inp))


@pytest.mark.parametrize("name", ["gn_tiny", "gn_c2_structure", "gn_gelu", "gn_bf16"])
def test_group_norm_two_pass_forced(cuda_lib, name):
    wl = SMALL[name]
    inp = _inputs(wl)
    ref, _ = oracle_full(wl, inp)
    y, am, path = run_gpu(cuda_lib, wl, inp, force_path=cuda_lib.PATH_TC_TWO_PASS)
    assert path == "tc_two_pass"
    compare(wl, y, am, ref, None, path, name)


@pytest.mark.parametrize("name,math", [("gn_c2_structure", 0), ("gn_bf16", 0), ("gn_cpg16", 3)])
def test_fused_gn_weights_change_between_calls(cuda_lib, name, math):
    # Every call packs its weights: a call with new weights must see them, and calls on weights
    # packed beforehand (C1N_FLAG_WEIGHTS_PACKED) must interleave with packing calls (the grid
    # exchange's epochs stay in step).
    wl = SMALL[name]
    inp = _inputs(wl)
    inp2 = dict(inp, w=(-0.5 * inp["w"][::-1]).copy())  # other weights, same shapes and scale
    ref1, _ = oracle_full(wl, inp)
    ref2, _ = oracle_full(wl, inp2)
    params = cuda_lib.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right,
                                  wl.dilation, wl.norm, wl.groups, wl.eps, wl.post, wl.dtype, math)
    op = cuda_lib.Conv1dNorm(params)
    assert op.path == "tc_fused_gn" and op.info.kernels == 2
    bf = wl.dtype == synth.DTYPE_BF16
    x, w1, w2 = _to_dev(inp["x"], bf), _to_dev(inp["w"], bf), _to_dev(inp2["w"], bf)
    b, ga, be = (_to_dev(inp[k], False) for k in ("b", "gamma", "beta"))
    tol = 1e-4 if math == 3 else None
    outs = []
    for w, packed in ((w1, False), (w2, False), (w1, False), (w2, True), (w2, False)):
        if packed:
            op.pack_weights(w1)  # the flag says: use what is packed (w1), not the w passed
        outs.append(op(x, w, b, ga, be, weights_packed=packed).float().cpu().numpy())
        op.check()
    compare(wl, outs[0], None, ref1, None, op.path, name + " (w1)", tol)
    compare(wl, outs[1], None, ref2, None, op.path, name + " (w2)", tol)
    np.testing.assert_array_equal(outs[2], outs[0])  # same inputs, same bits
    np.testing.assert_array_equal(outs[3], outs[0])  # pre-packed w1
    np.testing.assert_array_equal(outs[4], outs[1])
    # The same call captured once in a CUDA graph and replayed: new contents of the weight buffer
    # between replays must be packed and used.
    wbuf = w1.clone()
    y = torch.empty_like(op(x, wbuf, b, ga, be))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        op(x, wbuf, b, ga, be, out=y)
    for w, want in ((w2, outs[1]), (w1, outs[0]), (w2, outs[1])):
        wbuf.copy_(w)
        g.replay()
        torch.cuda.synchronize()
        op.check()
        np.testing.assert_array_equal(y.float().cpu().numpy(), want)
    op.close()


GN_NAMES = ["gn_tiny", "gn_c2_structure", "gn_cpg1", "gn_cpg4", "gn_cpg16", "gn_cpg25", "gn_cpg128", "gn_gelu",
            "gn_bf16", "gn_ragged_out"]


def _kernel_names(c1n, wl, inp, force_path, mainloop):
    params = c1n.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation,
                             wl.norm, wl.groups, wl.eps, wl.post, wl.dtype, 0, force_path, mainloop)
    op = c1n.Conv1dNorm(params)
    op.set_profiling(True)
    bf = wl.dtype == synth.DTYPE_BF16
    x, w = _to_dev(inp["x"], bf), _to_dev(inp["w"], bf)
    b, ga, be = (_to_dev(inp[k], False) for k in ("b", "gamma", "beta"))
    op(x, w, b, ga, be)
    torch.cuda.synchronize()
    op.check()
    return [n for n, _ in op.kernel_times()]


@pytest.mark.parametrize("name", GN_NAMES + ["gn_cb2", "gn_cb2_straddle", "gn_long_ragged", "gn_g1_twopass",
                                             "ln_c640_f32", "ln_c384_f32", "ln_gelu_bf16"])
@pytest.mark.parametrize("mode", ["single", "pair"])
def test_two_pass_epilogue_partials(cuda_lib, name, mode):
    # Two-pass plans: the conv epilogue writes the raw tile and its partial statistics, a small
    # kernel merges them (no pass re-reads the raw output for statistics) -- except GroupNorm whose
    # groups straddle a channel block, which keeps the statistics pass.
    wl = SMALL[name]
    inp = _inputs(wl)
    mainloop = cuda_lib.MAINLOOP_SINGLE if mode == "single" else cuda_lib.MAINLOOP_PAIR
    try:
        cuda_lib.conv1d_norm_destroy(cuda_lib.conv1d_norm_desc_create(cuda_lib.make_params(
            wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation, wl.norm,
            wl.groups, wl.eps, wl.post, wl.dtype, 0, cuda_lib.PATH_TC_TWO_PASS, mainloop)))
    except cuda_lib.C1NError:
        pytest.skip("plan cannot run on CTA pairs")
    ref, _ = oracle_full(wl, inp)
    y, am, path = run_gpu(cuda_lib, wl, inp, force_path=cuda_lib.PATH_TC_TWO_PASS, mainloop=mainloop)
    assert path == "tc_two_pass"
    compare(wl, y, am, ref, None, path, f"{name}/{mode}")
    names = _kernel_names(cuda_lib, wl, inp, cuda_lib.PATH_TC_TWO_PASS, mainloop)
    if wl.norm == synth.NORM_GROUP:
        assert names[-2] == ("gn_stats" if name == "gn_cb2_straddle" else "gn_merge"), names
    else:
        assert names[-2] == "ln_merge", names


@pytest.mark.parametrize("name", GN_NAMES)
def test_group_norm_cluster_exchange_forced(cuda_lib, name):
    # the same fused kernel with the partial statistics exchanged through a cluster's DSMEM
    wl = SMALL[name]
    inp = _inputs(wl)
    ref, _ = oracle_full(wl, inp)
    y, am, path = run_gpu(cuda_lib, wl, inp, force_path=cuda_lib.PATH_TC_FUSED_GN_DSMEM)
    assert path == "tc_fused_gn_dsmem"
    compare(wl, y, am, ref, None, path, name)


@pytest.mark.parametrize("name", ["ln_gelu_bf16", "ln_c384_f32"])
def test_layer_norm_two_pass_forced(cuda_lib, name):
    wl = SMALL[name]
    inp = _inputs(wl)
    ref, _ = oracle_full(wl, inp)
    y, am, path = run_gpu(cuda_lib, wl, inp, force_path=cuda_lib.PATH_TC_TWO_PASS)
    assert path == "tc_two_pass"
    compare(wl, y, am, ref, None, path, name)


@pytest.mark.parametrize("name", ["ln_gelu_bf16", "ln_c384_f32", "ln_c512_bf16"])
def test_layer_norm_fused_forced(cuda_lib, name):
    # the whole channel row of a tile (up to 512 channels) normalized in the tensor-core epilogue
    wl = SMALL[name]
    inp = _inputs(wl)
    ref, _ = oracle_full(wl, inp)
    y, am, path = run_gpu(cuda_lib, wl, inp, force_path=cuda_lib.PATH_TC_FUSED_LN)
    assert path == "tc_fused_ln"
    compare(wl, y, am, ref, None, path, name)


@pytest.mark.parametrize("name,path,kernels", [("gn_tiny", -1, ["pack_weights", "tc_conv"]),  # grid exchange
                                               ("gn_tiny", 5, ["pack_weights", "tc_conv"]),  # cluster exchange
                                               ("ln_c384_f32", 3, ["pack_weights", "tc_conv", "ln_merge", "normalize"]),
                                               ("linear_rowmin", -1, ["tc_conv", "rowmin_finish"]),
                                               ("stride2_simt", -1, ["simt_conv", "gn_stats", "normalize"])])
def test_kernel_times_list_every_launch(cuda_lib, name, path, kernels):
    # the profiling hook reports each kernel one run launches, in order, with its device time
    wl = SMALL[name]
    inp = _inputs(wl)
    params = cuda_lib.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right,
                                  wl.dilation, wl.norm, wl.groups, wl.eps, wl.post, wl.dtype,
                                  cuda_lib.MATH_SIMT if name in TC_REFUSED else 0, path)
    op = cuda_lib.Conv1dNorm(params)
    op.set_profiling(True)
    x, w = _to_dev(inp["x"], False), _to_dev(inp["w"], False)
    b, ga, be, b2 = (_to_dev(inp[k], False) for k in ("b", "gamma", "beta", "bias2"))
    out = torch.empty((wl.N, wl.C_out, op.T_out), dtype=op.out_dtype(), device="cuda")
    am = torch.empty((wl.N, op.T_out), dtype=torch.int32, device="cuda") if wl.post == synth.POST_ROWMIN_BIAS else None
    op(x, w, b, ga, be, bias2=b2, out=out, argmin=am)
    times = op.kernel_times()
    assert [n for n, _ in times] == kernels
    assert len(times) == op.info.kernels
    assert all(ms > 0 for _, ms in times)
    op.check()


def test_gelu_accuracy_on_exact_inputs(cuda_lib):
    # Linear with identity weights and no bias: the GEMM reproduces x exactly (x on a grid of 1/64
    # steps is exact in tf32), so the output differs from the oracle's float64 exact-erf GELU by the
    # kernel's GELU alone.
    wl = synth.LINEAR_GN_ROWMIN.replace(N=384, C_in=64, C_out=64, norm=synth.NORM_NONE, post=synth.POST_GELU_ERF)
    grid = (np.arange(wl.N * wl.C_in, dtype=np.float64) % 769 - 384) / 64.0  # -6 .. 6
    inp = {"x": grid.astype(np.float32).reshape(wl.N, wl.C_in, 1), "w": np.eye(64, dtype=np.float32)[:, :, None],
           "b": np.zeros(64, np.float32), "gamma": None, "beta": None, "bias2": None}
    ref, _ = oracle_full(wl, inp)
    y, _, path = run_gpu(cuda_lib, wl, inp)
    assert path == "tc_linear"
    err = np.abs(y.astype(np.float64) - ref)
    assert err.max() < 3e-6, err.max()


X3_NAMES = ["gn_tiny", "gn_c2_structure", "gn_cpg4", "gn_gelu", "gn_ragged_out", "causal_k4", "conv_dil3_pads",
            "conv_k1", "conv_gelu", "ln_c384_f32"]


@pytest.mark.parametrize("name", X3_NAMES)
def test_tensor_x3_meets_fp32_tolerance(cuda_lib, name):
    # 3xTF32 (head + tail split of both operands, three MMAs per step): the tensor-core path held to
    # the fp32 tolerance of the SIMT check path
    wl = SMALL[name]
    inp = _inputs(wl)
    ref, _ = oracle_full(wl, inp)
    y, am, path = run_gpu(cuda_lib, wl, inp, math=cuda_lib.MATH_TENSOR_X3)
    assert path != "simt"
    compare(wl, y, am, ref, None, path, name + " (3xTF32)", tol=TOL_SIMT)


def test_tensor_x3_full_conv_gn(cuda_lib):
    wl = synth.CONV_GN
    inp = _inputs(wl)
    ref, _ = oracle_full(wl, inp)
    y, _, path = run_gpu(cuda_lib, wl, inp, math=cuda_lib.MATH_TENSOR_X3)
    assert path == "tc_fused_gn"
    compare(wl, y, None, ref, None, path, wl.name + " (3xTF32)", tol=TOL_SIMT)


def test_repeated_calls_are_identical(cuda_lib):
    wl = SMALL["gn_c2_structure"]
    inp = _inputs(wl)
    y1, _, _ = run_gpu(cuda_lib, wl, inp)
    y2, _, _ = run_gpu(cuda_lib, wl, inp)
    assert np.array_equal(y1, y2)


# ------------------------------------------------------------------------------ the five workloads

def test_conv_gn_tiny_full(cuda_lib):
    wl = synth.CONV_GN_TINY
    inp = _inputs(wl)
    ref, _ = oracle_full(wl, inp)
    y, _, path = run_gpu(cuda_lib, wl, inp)
    assert path == "tc_fused_gn"
    compare(wl, y, None, ref, None, path, wl.name)


def test_conv_gn_full(cuda_lib):
    wl = synth.CONV_GN
    inp = _inputs(wl)
    ref, _ = oracle_full(wl, inp)
    y, _, path = run_gpu(cuda_lib, wl, inp)
    assert path == "tc_fused_gn"
    compare(wl, y, None, ref, None, path, wl.name)
    y_dsmem, _, path = run_gpu(cuda_lib, wl, inp, force_path=cuda_lib.PATH_TC_FUSED_GN_DSMEM)
    compare(wl, y_dsmem, None, ref, None, path, wl.name + " (cluster exchange)")
    # with gamma = 1, beta = 0 every (n, group) of the output has mean ~0 and variance ~1
    inp2 = dict(inp, gamma=None, beta=None)
    y2, _, _ = run_gpu(cuda_lib, wl, inp2)
    g = y2.reshape(wl.N, wl.groups, -1).astype(np.float64)
    assert np.max(np.abs(g.mean(axis=2))) < 1e-3
    assert np.max(np.abs(g.var(axis=2) - 1.0)) < 1e-2


def test_chained_calls_read_the_producers_output(cuda_lib):
    # Two fused-GroupNorm calls on one stream, the first one's y being the second one's x, as in
    # stacked layers. Each conv kernel lets the next kernel launch once its MMAs are done, before
    # its epilogue has stored y, and at this size the weight pack lets the second conv launch before
    # the pack itself waits: the second conv must still read the finished y. Its output must equal,
    # bit for bit, the same call made after a full synchronisation, eagerly and in a CUDA graph.
    wl_b = synth.CONV_GN
    wl_a = synth.Workload("chain_producer_n16_c64x128_t1024", N=wl_b.N, C_in=64, C_out=wl_b.C_in, T=wl_b.T, k=3,
                          pad_left=1, pad_right=1, norm=synth.NORM_GROUP, groups=16)
    ops, dev = [], []
    for wl in (wl_a, wl_b):
        params = cuda_lib.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right,
                                      wl.dilation, wl.norm, wl.groups, wl.eps, wl.post, wl.dtype, 0)
        op = cuda_lib.Conv1dNorm(params)
        assert op.path == "tc_fused_gn"
        inp = _inputs(wl)
        ops.append(op)
        dev.append({k: _to_dev(inp[k], False) for k in ("x", "w", "b", "gamma", "beta")})
    op_a, op_b = ops
    a, b = dev
    y_a = torch.empty((wl_a.N, wl_a.C_out, op_a.T_out), device="cuda")
    y_b = torch.empty((wl_b.N, wl_b.C_out, op_b.T_out), device="cuda")

    def chain():
        op_a(a["x"], a["w"], a["b"], a["gamma"], a["beta"], out=y_a)
        op_b(y_a, b["w"], b["b"], b["gamma"], b["beta"], out=y_b)

    chain()
    torch.cuda.synchronize()
    op_a.check()
    op_b.check()
    x_b = y_a.clone()
    torch.cuda.synchronize()
    want = op_b(x_b, b["w"], b["b"], b["gamma"], b["beta"])
    torch.cuda.synchronize()
    assert torch.equal(y_b, want)
    for _ in range(3):  # again, behind other work, eagerly
        y_a.fill_(float("nan"))
        y_b.fill_(float("nan"))
        chain()
    torch.cuda.synchronize()
    assert torch.equal(y_a, x_b) and torch.equal(y_b, want)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for _ in range(3):
        y_a.fill_(float("nan"))
        y_b.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        op_a.check()
        op_b.check()
        assert torch.equal(y_a, x_b) and torch.equal(y_b, want)


def test_causal_conv_full_sampled(cuda_lib):
    wl = synth.CAUSAL_CONV
    inp = _inputs(wl)
    y, _, path = run_gpu(cuda_lib, wl, inp)  # AUTO: CTA pairs at this size
    assert path == "tc_direct"
    y1, _, _ = run_gpu(cuda_lib, wl, inp, mainloop=cuda_lib.MAINLOOP_SINGLE)
    # 8 samples spread over the batch: the persistent CTAs (one per SM) walk 2048 tiles, so these
    # samples' tiles fall in the first, middle and last work units of the schedule
    ns = [0, 4, 9, 13, 18, 22, 27, wl.N - 1]
    ref, _ = oracle.conv1d_norm_samples(oracle.params_of(wl), ns, inp["x"], inp["w"], inp["b"])
    compare(wl, y[ns], None, ref, None, path, wl.name)
    compare(wl, y1[ns], None, ref, None, path, wl.name + " (one CTA per tile)")
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(y1))


def test_linear_gn_rowmin_full_sampled(cuda_lib):
    wl = synth.LINEAR_GN_ROWMIN
    inp = _inputs(wl)
    y, am, path = run_gpu(cuda_lib, wl, inp)
    assert path == "tc_linear"
    # one row from each of the eight 128-row M tiles (the CTA pairs take 256-row tiles)
    ns = [5, 130, 300, 420, 555, 700, 833, wl.N - 1]
    p = oracle.params_of(wl)
    ref, ref_am = oracle.conv1d_norm_samples(p, ns, inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"],
                                             inp["bias2"])
    compare(wl, y[ns], None, ref, None, path, wl.name)
    check_argmin(am[ns], ref_am, _argmin_margin(wl, inp, ns))
    # every row is its minimum plus the broadcast bias
    b2 = inp["bias2"].astype(np.float64)
    rows = y[:, :, 0].astype(np.float64) - b2[None, :]
    assert np.max(np.abs(rows - rows[:, :1])) < 1e-5


def test_conv_ln_gelu_bf16_full_sampled(cuda_lib):
    wl = synth.CONV_LN_GELU_BF16
    inp = _inputs(wl)
    y, _, path = run_gpu(cuda_lib, wl, inp)
    assert path == "tc_fused_ln"
    y2, _, path2 = run_gpu(cuda_lib, wl, inp, force_path=cuda_lib.PATH_TC_TWO_PASS)
    assert path2 == "tc_two_pass"
    ns = [0, 9, 18, 27, 36, 45, 54, wl.N - 1]  # spread over the persistent clusters' schedule
    ref, _ = oracle.conv1d_norm_samples(oracle.params_of(wl), ns, inp["x"], inp["w"], inp["b"], inp["gamma"],
                                        inp["beta"])
    compare(wl, y[ns], None, ref, None, path, wl.name)
    compare(wl, y2[ns], None, ref, None, path2, wl.name + " (two-pass)")
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(y2))
