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


def _args(**kw):
    ns = argparse.Namespace(micro_batch_size=31, sequence_length=512, hidden_size=4096, intermediate_size=16384,
                            parallel="replicas")
    for k, v in kw.items():
        setattr(ns, k, v)
    return ns


def test_both_arms_print_the_same_config():
    """The reference arm and the product arm build `config` with one function."""
    a = bench.contract_config(_args(), 1, "nvfp4", True)
    assert a == bench.contract_config(_args(), 1, "nvfp4", True)
    assert a["workload"].startswith("CodonFM-5B layer, 12 GEMMs, nvfp4 autocast (M=15872")
    assert a["global_batch"] == 31 and a["parallelism"] == "replicas x1"
    t = bench.contract_config(_args(parallel="tokens"), 4, "nvfp4", True)
    assert t["global_batch"] == 124 and t["parallelism"].startswith("token-sharded data parallel")


def test_quantizer_bytes_per_layer():
    """Per-GEMM autocast quantizes one copy of each GEMM operand: 2.483 G
    operand elements per CodonFM-5B layer, x 4.5625 B for NVFP4 (amax pass 2,
    read 2, E2M1 codes 0.5, E4M3 scales 1/16)."""
    layer = bench.Layer.__new__(bench.Layer)
    h, f, M = 4096, 16384, 15872
    layer.shapes = []
    for name, K, N in (("qkv", h, 3 * h), ("attn_out", h, h), ("mlp_up", h, f), ("mlp_down", f, h)):
        layer.shapes += [(name + "_fprop", 0, M, K, N), (name + "_dgrad", 1, M, N, K), (name + "_wgrad", 2, N, M, K)]
    elems = sum(m * k + n * k for _, _, m, k, n in layer.shapes)
    assert elems == 2_483_027_968
    assert bench.quant_bytes_per_layer(layer, "nvfp4") == pytest.approx(elems * 4.5625)
    assert bench.quant_bytes_per_layer(layer, "fp8_delayed") == pytest.approx(elems * 3)
    assert bench.quant_bytes_per_layer(layer, "bf16") == 0


def test_dp_kernels_per_step():
    """Token-sharded step per linear: W amax + tile pass, the X and dY amax
    passes, their tile passes and three GEMMs (NVFP4); MX formats have no
    amax passes."""
    assert bench.dp_kernels_per_step("nvfp4") == 4 * 9
    assert bench.dp_kernels_per_step("mxfp8") == 4 * 6
    assert bench.dp_kernels_per_step("bf16") == 4 * 3
