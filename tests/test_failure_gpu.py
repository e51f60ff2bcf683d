"""Device failure path, exercised without faulting or hanging the GPU: a bounded wait is made to run
out on purpose and the kernel must return, report C1N_ERR_TIMEOUT through conv1d_norm_check and
leave the workspace usable for the next run.

With C1N_FLAG_TEST_STALL_EXCHANGE the first CTA of the fused GroupNorm grid exchange withholds its
partial statistics, so the other CTAs of its sample wait for words that nothing writes; every such
wait gives up after about one second of %globaltimer and the kernel finishes normally."""
import time

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

WL = synth.CONV_GN.replace(N=2, C_in=32, C_out=64, T=512, groups=8)  # 2 samples x 4 time tiles


def _setup(c1n, wl):
    inp = synth.make_inputs(wl, seed=11)
    dev = {k: (None if v is None else torch.from_numpy(v).cuda()) for k, v in inp.items()}
    params = c1n.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right, wl.dilation,
                             wl.norm, wl.groups, wl.eps, wl.post, wl.dtype)
    return dev, c1n.Conv1dNorm(params)


def _args(c1n, dev, y, flags):
    p = lambda t: None if t is None else t.data_ptr()
    return c1n.Args(p(dev["x"]), p(dev["w"]), p(dev["b"]), p(dev["gamma"]), p(dev["beta"]), None, y.data_ptr(), None,
                    None, 0, flags)


def test_stalled_exchange_times_out_and_the_next_run_recovers(cuda_lib):
    c1n = cuda_lib
    dev, op = _setup(c1n, WL)
    assert op.path == "tc_fused_gn"
    stream = torch.cuda.current_stream().cuda_stream
    y_ref = op(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"])
    torch.cuda.synchronize()
    op.check()

    y = torch.empty_like(y_ref)
    t0 = time.perf_counter()
    c1n.conv1d_norm_run_ex(op.desc, _args(c1n, dev, y, c1n.FLAG_TEST_STALL_EXCHANGE), stream)
    torch.cuda.synchronize()  # the kernel returns on its own once its waits give up
    elapsed = time.perf_counter() - t0
    assert 0.5 < elapsed < 10.0, elapsed
    with pytest.raises(c1n.C1NError) as e:
        op.check()
    assert e.value.status == c1n.ERR_TIMEOUT
    assert "site 10" in str(e.value)  # the grid-exchange wait
    op.check()  # the status word was cleared

    # the workspace is usable again: with the pack, and with the weights already packed
    for packed in (False, True):
        y2 = op(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"], weights_packed=packed)
        torch.cuda.synchronize()
        op.check()
        assert torch.equal(y2, y_ref), f"weights_packed={packed}"


def test_stall_flag_needs_the_grid_exchange_plan(cuda_lib):
    c1n = cuda_lib
    wl = synth.CAUSAL_CONV.replace(N=1, C_in=32, C_out=32, T=256)  # no GroupNorm: nothing to withhold
    dev, op = _setup(c1n, wl)
    y = torch.empty((wl.N, wl.C_out, op.T_out), device="cuda")
    with pytest.raises(c1n.C1NError) as e:
        c1n.conv1d_norm_run_ex(op.desc, _args(c1n, dev, y, c1n.FLAG_TEST_STALL_EXCHANGE),
                               torch.cuda.current_stream().cuda_stream)
    assert e.value.status == c1n.ERR_INVALID_ARG
    np.testing.assert_array_equal(np.array([op.path]), np.array(["tc_direct"]))
