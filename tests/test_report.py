"""The speed-up analysis tables of bench.py --workload report, checked on CPU
against the worked example the pages print ([TE], 'interpreting real-model
results': per-shape NVFP4 vs MXFP8 Fprop times on B300 and their blended
ratio), and on hand-made inputs for the below-BF16 diagnostic."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "codonfm5b_layer.json")))
LINEARS = ["qkv", "attn_out", "mlp_up", "mlp_down"]
SHAPES = [(f"{lin}_{p}", i, 1, 1, 1) for lin in LINEARS for i, p in enumerate(("fprop", "dgrad", "wgrad"))]


def times(recipe, fprop_only=None, other=1.0):
    t = {n: other for n, *_ in SHAPES}
    for lin, v in (fprop_only or {}).items():
        t[f"{lin}_fprop"] = v
    return {"autocast": dict(t), "prequant": dict(t)}


def test_pages_fprop_ratios_and_blend():
    per = {r: times(r, {lin: GOLD["fprop_ms_b300"][lin][r] for lin in LINEARS}) for r in ("mxfp8", "nvfp4")}
    out, lines = bench.report_tables(per, SHAPES, LINEARS)
    ratios = out["nvfp4_vs_mxfp8"]["autocast"]
    for lin in LINEARS:
        assert round(ratios[f"{lin}_fprop"], 2) == GOLD["fprop_ms_b300"][lin]["ratio"]
    assert round(ratios["blended_fprop"], 2) == GOLD["blended_fprop_ratio"]
    assert any("NVFP4 vs MXFP8 Fprop" in ln for ln in lines)


def test_below_bf16_lists_only_slower_shapes():
    bf = times("bf16")
    bf["autocast"] = {n: 1.1 for n in bf["autocast"]}  # the slower BF16 run is not the baseline
    per = {"bf16": bf, "nvfp4": times("nvfp4", {"attn_out": 1.25}, other=0.5)}
    out, lines = bench.report_tables(per, SHAPES, LINEARS)
    assert out["below_bf16"] == ["nvfp4/autocast/attn_out_fprop", "nvfp4/prequant/attn_out_fprop"]
    assert out["speedup_vs_bf16"]["nvfp4"]["prequant"]["qkv_fprop"] == 2.0
    assert out["dgrad_vs_fprop"]["nvfp4"]["attn_out"] == 0.5 / 1.25
    assert lines[-1].startswith("below BF16: nvfp4/autocast/attn_out_fprop")


def test_projection_and_step_diagnostic():
    """End-to-end projection: the layer's GEMM times (autocast: with their
    quantization) x the layer count, and the pages' three readings of the
    GEMM-only speed-up against the step's (about equal: the GEMMs dominate;
    much larger: work outside the GEMMs eats the gain; below 1: not faster)."""
    base = times("bf16")                                            # 12 ms per layer
    per = {"bf16": base,
           "dominant": {"autocast": {n: 0.55 for n, *_ in SHAPES}, "prequant": {n: 0.5 for n, *_ in SHAPES}},
           "overhead": {"autocast": {n: 0.9 for n, *_ in SHAPES}, "prequant": {n: 0.3 for n, *_ in SHAPES}},
           "slower": {"autocast": {n: 1.3 for n, *_ in SHAPES}, "prequant": {n: 1.2 for n, *_ in SHAPES}}}
    out, lines = bench.report_tables(per, SHAPES, LINEARS, layers=24)
    p = out["projection"]["recipes"]
    assert out["projection"]["layers"] == 24
    assert p["dominant"]["gemm_only_speedup"] == pytest.approx(2.0)
    assert p["dominant"]["step_speedup"] == pytest.approx(1 / 0.55)
    assert p["dominant"]["model_ms"]["autocast"] == pytest.approx(24 * 12 * 0.55)
    assert "GEMMs dominate" in p["dominant"]["diagnostic"]
    assert "consumes the gain" in p["overhead"]["diagnostic"]      # 3.33x GEMM-only vs 1.11x step
    assert "below 1.0" in p["slower"]["diagnostic"]
    assert p["bf16"]["diagnostic"] == "the baseline"
    assert any(ln.startswith("overhead: GEMM-only 3.33x, step 1.11x, 24 layers") for ln in lines)
