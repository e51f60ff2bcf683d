"""Host-side logic of bench.py, without a GPU: which roofline bounds a workload and which measured
peak it is held to, and when a committed DRAM-traffic record applies."""
import json
import types

import pytest

import bench
import synth

PEAKS = {"hbm_gbs": 6684.5, "bf16_tflops": 1928.5, "bf16_tflops_sustained": 1747.8, "source": "measured"}


def _run(wl, path):
    bf = wl.dtype == synth.DTYPE_BF16
    return types.SimpleNamespace(path=path, bf=bf, kernels=2, kernels_packed=1)


def test_conv_gn_is_held_to_hbm_and_tensor_workloads_to_the_sustained_peak():
    # conv_gn: 25.6 MB and 3.22 GFLOP -> the bytes take longer at the measured peaks: HBM-bound
    wl = synth.CONV_GN
    r = bench.conv_roofline(wl, _run(wl, "tc_fused_gn"), PEAKS, {}, 0.018)
    assert r["bound"] == "hbm" and r["peak"] == PEAKS["hbm_gbs"] and r["peak_kind"] == "copy bandwidth"
    assert r["achieved"] == pytest.approx(wl.algorithmic_bytes / 0.018e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["hbm_gbs"])
    # causal_conv (TF32) and the bf16 LayerNorm: tensor-bound, against the sustained figure
    for wl, path, ratio in ((synth.CAUSAL_CONV, "tc_direct", bench.TF32_PER_BF16),
                            (synth.CONV_LN_GELU_BF16, "tc_fused_ln", 1.0)):
        r = bench.conv_roofline(wl, _run(wl, path), PEAKS, {}, 0.2)
        assert r["bound"] == "tensor" and r["peak_kind"].startswith("sustained")
        assert r["peak"] == pytest.approx(PEAKS["bf16_tflops_sustained"] * ratio)
        assert r["frac_of_burst_peak"] == pytest.approx(r["frac"] * PEAKS["bf16_tflops_sustained"] /
                                                        PEAKS["bf16_tflops"])


def test_two_pass_plans_count_the_raw_tile_instead_of_y():
    wl = synth.CONV_LN_GELU_BF16  # bf16 y; the two-pass conv writes an fp32 raw tile
    one = bench.conv_roofline(wl, _run(wl, "tc_fused_ln"), PEAKS, {}, 0.3)
    two = bench.conv_roofline(wl, _run(wl, "tc_two_pass"), PEAKS, {"normalize": 0.16, "tc_conv": 0.26}, 0.3)
    y = wl.N * wl.C_out * wl.T_out
    assert two["algorithmic_bytes"] - one["algorithmic_bytes"] == y * (4 - wl.elem_bytes)


def test_traffic_record_applies_only_to_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    from gemm_groupnorm_accelerator_gb300 import _build_lib
    rec = {"path": "tc_fused_gn", "source_file": "tc_conv.cu",
           "source_fingerprint": _build_lib.kernel_fingerprint("tc_conv.cu"), "dram_bytes_per_launch": 123}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({synth.CONV_GN.name: rec}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic(synth.CONV_GN.name, "tc_fused_gn") == 123
    assert bench.read_traffic(synth.CONV_GN.name, "tc_two_pass") is None  # another plan
    rec["source_fingerprint"] = "0" * 64  # taken on other sources
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({synth.CONV_GN.name: rec}))
    assert bench.read_traffic(synth.CONV_GN.name, "tc_fused_gn") is None

