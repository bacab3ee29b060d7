"""The benchmark's host-side arithmetic (CPU only): roofline peaks, the epilogue floor, the
whole-job throughput, the profile-summary names and which sources the traffic figures are
tied to."""
import math
import os

import pytest

import bench
import fc_inputs

PK = {"hbm_gbs": 6774.2, "bf16_tflops": 1911.6, "bf16_tflops_sustained": 1723.9, "source": "measured"}


def test_tensor_peaks_per_precision():
    tf32 = PK["bf16_tflops"] * 1.1 / 2.25
    assert bench.tensor_peak(fc_inputs.WORKLOADS["B"], PK)[0] == pytest.approx(tf32)
    assert bench.tensor_peak(fc_inputs.WORKLOADS["E"], PK)[0] == pytest.approx(PK["bf16_tflops"])
    assert bench.tensor_peak(fc_inputs.WORKLOADS["B3"], PK)[0] == pytest.approx(tf32 / 3)
    assert bench.tensor_peak(fc_inputs.WORKLOADS["D3"], PK)[0] == pytest.approx(tf32 / 3)
    assert bench.tensor_peak(fc_inputs.WORKLOADS["Db"], PK)[0] == pytest.approx(PK["bf16_tflops"])


def test_tf32_peak_is_the_larger_of_nominal_and_measured():
    nominal = PK["bf16_tflops"] * 1.1 / 2.25
    pk = dict(PK, tf32_measured_tflops=1022.2, tf32_how="test")
    peak, note = bench.tf32_peak(pk)
    assert peak == pytest.approx(1022.2) and "measured" in note
    assert bench.tensor_peak(fc_inputs.WORKLOADS["B"], pk)[0] == pytest.approx(1022.2)
    assert bench.tensor_peak(fc_inputs.WORKLOADS["B3"], pk)[0] == pytest.approx(1022.2 / 3)
    assert bench.tensor_peak(fc_inputs.WORKLOADS["E"], pk)[0] == pytest.approx(PK["bf16_tflops"])   # bf16: unchanged
    low = dict(PK, tf32_measured_tflops=500.0, tf32_how="test")
    assert bench.tf32_peak(low)[0] == pytest.approx(nominal)
    assert bench.tf32_peak(PK)[0] == pytest.approx(nominal)                                          # not measured


def test_round_to_four_significant_digits():
    assert bench.r4(0.23412345) == 0.2341 and bench.r4(1234.5678) == 1235.0 and bench.r4(None) is None


def test_workload_b_roofline_figures():
    wl = fc_inputs.WORKLOADS["B"]
    assert wl.flops() == 2 * 128 * 64 * 254 * 254 * 8 * 9
    assert wl.compulsory_bytes() == 268486912
    t_tensor = wl.flops() / (bench.tensor_peak(wl, PK)[0] * 1e12)
    assert t_tensor * 1e6 == pytest.approx(81.4, abs=0.1)


def test_epilogue_floor_is_the_busier_unit():
    wl = fc_inputs.WORKLOADS["B"]
    r = bench.epilogue_roofline(wl, 0.316, 152, 2070.0)
    fma, sfu = bench.EPILOGUE_COST["gelu"]
    assert fma / 128 > sfu                                    # erf-GELU: the FMA pipe binds
    assert r["peak"] == pytest.approx(152 * 2070e6 * 128 / fma / 1e9)
    assert r["elements"] == 128 * 64 * 254 * 254
    assert r["achieved"] == pytest.approx(r["elements"] / 0.316e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    # Mish twice: two exponentials and two reciprocals per element bind the SFU
    fma2, sfu2 = bench.EPILOGUE_COST["mish_mish"]
    assert sfu2 > fma2 / 128
    rc = bench.epilogue_roofline(fc_inputs.WORKLOADS["C"], 1.0, 152, 2000.0)
    assert rc["peak"] == pytest.approx(152 * 2000e6 / sfu2 / 1e9)


def test_whole_job_throughput_counts_every_rank():
    assert bench.job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)
    assert bench.job_tflops(1e12, 4, 1.0) == pytest.approx(4000.0)


def test_profile_names_follow_kernel_and_workload():
    assert bench.traffic_profile_name("B") == \
        "conv3x3_fused_conv3x3_gelu_avgpool_f32_128x8x256x256_c64_dram_traffic.md"
    assert bench.traffic_profile_name("D").startswith("linear_lse_")


def test_host_only_sources_do_not_move_the_kernel_hash(tmp_path, monkeypatch):
    """Editing the host-buffer pipeline (no device code) keeps the traffic figures valid; editing a
    kernel source invalidates them."""
    csrc = tmp_path / "gemm_activation_reduction_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "fc_host.cu").write_text("host only\n")
    (csrc / "fc_conv.cu").write_text("__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_sources_hash()
    (csrc / "fc_host.cu").write_text("host only, edited\n")
    assert bench.kernel_sources_hash() == h0
    (csrc / "fc_conv.cu").write_text("__global__ void k() { }\n")
    assert bench.kernel_sources_hash() != h0


def test_inputs_smaller_than_l2_are_rotated_over_copies_twice_its_size():
    k3e = fc_inputs.WORKLOADS["K3e"].compulsory_bytes()          # 1024 x 8192 fp32 rows, 33.6 MB
    n = bench.rotation_copies(k3e)
    assert n == 8 and n * k3e >= 2 * bench.L2_BYTES > (n - 1) * k3e
    assert bench.rotation_copies(fc_inputs.WORKLOADS["K1e"].compulsory_bytes()) == 1   # 2.1 GB: one copy
