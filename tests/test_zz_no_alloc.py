"""The entry point that allocates nothing, checked on the GPU against the regular entry point.

conv1d_norm_run_static_scratch serves callers that may not allocate device memory where they run
the operator (a host framework that owns every device allocation, a plugin that may not allocate
after start-up, a real-time loop that must not wait on an allocator). Instead of a caller-provided
workspace it uses a fixed array in the library's device image. This file is collected last so that
a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_TF32 = 5e-3  # the tensor-core fp32 tolerance the parity tests use


def _params(c1n, wl, force_path=-1):
    return c1n.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation,
                           wl.norm, wl.groups, wl.eps, wl.post, wl.dtype, force_path=force_path)


class _Case:
    """One operator: its inputs on the device, the regular entry point's output (run_ex with a
    caller-owned workspace) and a descriptor for the entry point without allocation."""

    def __init__(self, c1n, wl, seed):
        self.c1n, self.wl = c1n, wl
        self.inp = synth.make_inputs(wl, seed=seed)
        self.dev = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in self.inp.items()}
        params = _params(c1n, wl)
        op = c1n.Conv1dNorm(params)
        d = self.dev
        self.y_ref = op(d["x"], d["w"], d["b"], d["gamma"], d["beta"])
        torch.cuda.synchronize()
        op.check()
        self.path = op.path
        self.desc = c1n.conv1d_norm_desc_create(params)
        assert c1n.conv1d_norm_workspace_size(self.desc) <= c1n.STATIC_SCRATCH_BYTES

    def args(self, y, flags=0):
        d, p = self.dev, (lambda t: None if t is None else t.data_ptr())
        return self.c1n.Args(p(d["x"]), p(d["w"]), p(d["b"]), p(d["gamma"]), p(d["beta"]), None, y.data_ptr(), None,
                             None, 0, flags)

    def run_static(self):
        y = torch.full_like(self.y_ref, float("nan"))
        stream = torch.cuda.current_stream().cuda_stream
        self.c1n.conv1d_norm_run_static_scratch(self.desc, self.args(y), stream)
        torch.cuda.synchronize()
        self.c1n.conv1d_norm_check(self.desc, None, stream)
        return y

    def close(self):
        self.c1n.conv1d_norm_destroy(self.desc)


def test_static_scratch_matches_regular_entry_point_twice(cuda_lib):
    case = _Case(cuda_lib, synth.CONV_GN.replace(N=4), seed=3)
    try:
        ref, _ = oracle.conv1d_norm(oracle.params_of(case.wl), case.inp["x"], case.inp["w"], case.inp["b"],
                                    case.inp["gamma"], case.inp["beta"])
        for _ in range(2):
            y = case.run_static()
            # the same kernels on the same inputs: identical to the regular entry point, bit for bit
            assert torch.equal(y, case.y_ref)
            err = float(np.max(np.abs(y.cpu().numpy().astype(np.float64) - ref)))
            assert err <= TOL_TF32, err
    finally:
        case.close()


def test_static_scratch_alternating_descriptors(cuda_lib):
    # Two operators with different plans and workspace layouts share the one array; each call packs
    # its own weights, so alternating them leaves no trace of the other in either result.
    a = _Case(cuda_lib, synth.CONV_GN.replace(N=2, C_in=64, C_out=128, T=512, groups=16), seed=5)
    b = _Case(cuda_lib, synth.CAUSAL_CONV.replace(N=2, C_in=96, C_out=160, T=640), seed=6)
    try:
        assert a.path == "tc_fused_gn" and b.path == "tc_direct"
        for case in (a, b, a, b):
            assert torch.equal(case.run_static(), case.y_ref), case.wl.name
    finally:
        a.close()
        b.close()


def test_static_scratch_rejects_prepacked_weights(cuda_lib):
    c1n = cuda_lib
    case = _Case(c1n, synth.CONV_GN.replace(N=2), seed=7)
    try:
        y = torch.empty_like(case.y_ref)
        with pytest.raises(c1n.C1NError) as e:
            c1n.conv1d_norm_run_static_scratch(case.desc, case.args(y, flags=c1n.FLAG_WEIGHTS_PACKED),
                                               torch.cuda.current_stream().cuda_stream)
        assert e.value.status == c1n.ERR_INVALID_ARG
        assert torch.equal(case.run_static(), case.y_ref)  # a refused call leaves the next one intact
    finally:
        case.close()


def test_static_scratch_rejects_operators_that_need_more(cuda_lib):
    c1n = cuda_lib
    wl = synth.CONV_LN_GELU_BF16  # its two-pass plan keeps a raw fp32 copy of y in the workspace
    desc = c1n.conv1d_norm_desc_create(_params(c1n, wl, force_path=c1n.PATH_TC_TWO_PASS))
    try:
        assert c1n.conv1d_norm_workspace_size(desc) > c1n.STATIC_SCRATCH_BYTES
        buf = torch.zeros(16, dtype=torch.float32, device="cuda")
        p = buf.data_ptr()
        args = c1n.Args(p, p, None, None, None, None, p, None, None, 0, 0)
        with pytest.raises(c1n.C1NError) as e:
            c1n.conv1d_norm_run_static_scratch(desc, args, torch.cuda.current_stream().cuda_stream)
        assert e.value.status == c1n.ERR_WORKSPACE
        assert "fixed scratch" in str(e.value)
    finally:
        c1n.conv1d_norm_destroy(desc)
