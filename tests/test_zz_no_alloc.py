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

import synth

pytestmark = pytest.mark.gpu

TOL_TF32 = 5e-3  # the tensor-core fp32 tolerance the parity tests use


def _params(c1n, wl, force_path=-1):
    return c1n.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation,
                           wl.norm, wl.groups, wl.eps, wl.post, wl.dtype, force_path=force_path)


def test_static_scratch_matches_regular_entry_point_twice(cuda_lib):
    c1n = cuda_lib
    wl = synth.CONV_GN.replace(N=4)
    inp = synth.make_inputs(wl, seed=3)
    dev = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in inp.items()}
    params = _params(c1n, wl)
    op = c1n.Conv1dNorm(params)  # regular path: caller-owned workspace through run_ex
    y_ref = op(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"])
    torch.cuda.synchronize()
    op.check()

    desc = c1n.conv1d_norm_desc_create(params)
    try:
        assert c1n.conv1d_norm_workspace_size(desc) <= c1n.STATIC_SCRATCH_BYTES
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(2):
            y = torch.full_like(y_ref, float("nan"))
            args = c1n.Args(dev["x"].data_ptr(), dev["w"].data_ptr(), dev["b"].data_ptr(), dev["gamma"].data_ptr(),
                            dev["beta"].data_ptr(), None, y.data_ptr(), None, None, 0, 0)
            c1n.conv1d_norm_run_static_scratch(desc, args, stream)
            torch.cuda.synchronize()
            c1n.conv1d_norm_check(desc, None, stream)
            assert torch.isfinite(y).all()
            err = float((y.double() - y_ref.double()).abs().max())
            assert err <= TOL_TF32, err
    finally:
        c1n.conv1d_norm_destroy(desc)


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
