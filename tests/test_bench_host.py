"""CPU checks of the benchmark's host logic: recipe selection, the launch count
it claims, the clock-sample parsing, and that a DRAM-traffic figure is only
taken from a profile recorded for the kernel source as it stands."""
import argparse
import hashlib
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GEMM_CU = os.path.join(ROOT, "precision_transformer_gemms_gb300", "csrc", "gemm.cu")


def test_sweep_recipes_and_filters():
    ns = argparse.Namespace(no_fp8=False, no_fp4=False)
    assert bench.sweep_recipes(ns) == bench.RECIPES
    ns.no_fp8 = True
    assert not {"mxfp8", "mxfp8_e5m2"} & set(bench.sweep_recipes(ns))
    ns.no_fp4 = True
    assert bench.sweep_recipes(ns) == ["bf16", "fp8_delayed", "fp8_current"]


def test_kernels_per_step():
    """Launches of one layer step: 12 GEMMs, plus per quantized copy (24 per
    step) an amax pass and a tile pass where the format has a global amax."""
    layer = bench.Layer.__new__(bench.Layer)
    assert layer.kernels_per_step("bf16", True) == 12
    assert layer.kernels_per_step("nvfp4", False) == 12
    assert layer.kernels_per_step("nvfp4", True) == 12 + 48
    assert layer.kernels_per_step("mxfp8", True) == 12 + 24
    assert layer.kernels_per_step("mxfp4", True) == 12 + 24
    assert layer.kernels_per_step("fp8_current", True) == 12 + 48
    assert layer.kernels_per_step("fp8_delayed", False) == 12 + 48  # always dynamic


def test_clock_sampler_parsing():
    cs = bench.ClockSampler(0)
    cs.lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
                "0, 2055, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
                "0, 2070, 2070, 960.0, 0x0, Not Active, Not Active, Not Active, Not Active",
                "garbage"]
    out = cs.stop()
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    cs = bench.ClockSampler(0)
    cs.lines = ["0, 1500, 2070, 1000, 0x8, Active, Not Active, Active, Not Active"]
    out = cs.stop()
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and out["sm_mhz"] == 1500.0


def test_profiled_traffic_follows_the_kernel_source(tmp_path):
    """The committed profile is used only while gemm.cu hashes to the value it
    records; any other source (or a recipe without a profile) gives None."""
    path = os.path.join(ROOT, "profiles", "gemm_nvfp4_layer_traffic.md")
    text = open(path).read()
    sha = hashlib.sha256(open(GEMM_CU, "rb").read()).hexdigest()
    t = bench.profiled_traffic(GEMM_CU, "nvfp4")
    if sha in text:
        assert t is not None and t > 0
    else:
        assert t is None
    other = tmp_path / "gemm.cu"
    other.write_bytes(open(GEMM_CU, "rb").read() + b"\n// changed\n")
    assert bench.profiled_traffic(str(other), "nvfp4") is None
    assert bench.profiled_traffic(GEMM_CU, "no_such_recipe") is None


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(1.5, 1) == pytest.approx(1.5)
