"""The torch wrappers refuse tensors that do not match the operator before any pointer crosses the C
ABI (the library sees raw pointers only: a tensor of the wrong size would become out-of-bounds
device accesses, not an error status). Runs without a GPU: the descriptor is host-only and the
checks read tensor metadata."""
import pytest
import torch

import gemm_groupnorm_accelerator_gb300 as c1n
import synth


def _op(wl):
    params = c1n.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation,
                             wl.norm, wl.groups, wl.eps, wl.post, wl.dtype)
    return c1n.Conv1dNorm(params, device="meta")  # no device memory: the workspace is a meta tensor


def _good(wl, T_out, dtype=torch.float32):
    t = lambda *s, dt=dtype: torch.zeros(*s, dtype=dt)
    return dict(x=t(wl.N, wl.C_in, wl.T), w=t(wl.C_out, wl.C_in, wl.k), b=t(wl.C_out, dt=torch.float32),
                gamma=t(wl.C_out, dt=torch.float32), beta=t(wl.C_out, dt=torch.float32),
                bias2=t(wl.C_out, dt=torch.float32) if wl.post == synth.POST_ROWMIN_BIAS else None,
                out=t(wl.N, wl.C_out, T_out), argmin=None)


@pytest.mark.parametrize("wl", [synth.CONV_GN_TINY, synth.CONV_LN_GELU_BF16.replace(N=2, T=64),
                                synth.LINEAR_GN_ROWMIN.replace(N=8, C_in=64, C_out=64, groups=4)],
                         ids=lambda w: w.name)
def test_conv1d_norm_arguments_are_checked(wl):
    op = _op(wl)
    try:
        dt = torch.bfloat16 if wl.dtype == synth.DTYPE_BF16 else torch.float32
        good = _good(wl, op.T_out, dt)
        op.validate(**good)  # matching tensors pass
        bad_cases = [
            ("x", torch.zeros(wl.N, wl.C_in, wl.T + 1, dtype=dt)),          # wrong length
            ("x", torch.zeros(wl.N, wl.C_in, wl.T, dtype=torch.float64)),   # wrong dtype
            ("x", torch.zeros(wl.N, wl.C_in, 2 * wl.T, dtype=dt)[:, :, ::2]),  # not dense
            ("w", torch.zeros(wl.C_out, wl.C_in + 1, wl.k, dtype=dt)),
            ("b", torch.zeros(wl.C_out + 1)),
            ("gamma", torch.zeros(wl.C_out, dtype=torch.float16)),
            ("beta", torch.zeros(1, wl.C_out)),
            ("out", torch.zeros(wl.N, wl.C_out, op.T_out + 1, dtype=dt)),
            ("argmin", torch.zeros(wl.N, op.T_out, dtype=torch.int64)),
        ]
        for name, t in bad_cases:
            args = dict(good, **{name: t})
            with pytest.raises(ValueError, match=name):
                op.validate(**args)
            with pytest.raises(ValueError, match=name):  # the call checks before it runs anything
                op(**args)
        with pytest.raises(ValueError, match="w"):
            op.pack_weights(torch.zeros(wl.C_out, wl.C_in, wl.k + 1, dtype=dt))
        if wl.post == synth.POST_ROWMIN_BIAS:
            with pytest.raises(ValueError, match="bias2 is required"):
                op.validate(**dict(good, bias2=None))
    finally:
        op.close()


def test_conv1d_norm_tensors_must_share_the_workspace_device(monkeypatch):
    wl = synth.CONV_GN_TINY
    op = _op(wl)
    try:
        monkeypatch.setattr(op, "_device", lambda: torch.device("cuda", 0))
        with pytest.raises(ValueError, match="x is on cpu"):
            op.validate(**_good(wl, op.T_out))
    finally:
        op.close()


def test_p4_wrappers_check_their_tensors():
    x = torch.zeros(2, 32, 3, 4, 32)
    w = torch.zeros(32, 64, 3, 3, 3)
    with pytest.raises(ValueError, match="5-D"):
        c1n.conv_transpose3d(x[0], w)
    with pytest.raises(ValueError, match="w has shape"):
        c1n.conv_transpose3d(x, torch.zeros(32, 64, 3, 3, 2))
    with pytest.raises(ValueError, match="dtype"):
        c1n.conv_transpose3d(x.double(), w)
    with pytest.raises(ValueError, match="CUDA"):
        c1n.conv_transpose3d(x, w)
    with pytest.raises(ValueError, match="CUDA"):
        c1n.conv_transpose3d_ln_avgpool3d_gelu(x, w, None, 1.0)
    with pytest.raises(ValueError, match="5-D"):
        c1n.ln_avgpool3d_gelu(torch.zeros(2, 3, 4, 64), 1.0)
    with pytest.raises(ValueError, match="dtype"):
        c1n.ln_avgpool3d_gelu(torch.zeros(2, 3, 4, 4, 64, dtype=torch.float64), 1.0)
    with pytest.raises(ValueError, match="CUDA"):
        c1n.ln_avgpool3d_gelu(torch.zeros(2, 3, 4, 4, 64), 1.0)
