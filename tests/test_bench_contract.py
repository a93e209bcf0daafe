"""The reference arm of bench.py on the CPU: one JSON line with the keys the
benchmark contract names, the oracle timed on a bounded sample."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_flatten_sections_keeps_scalars():
    """Every configured workload's figure lands in flat scalar keys (top level and in
    the `prefill` dict), with each section's clock record beside it."""
    sys.path.insert(0, ROOT)
    import bench
    shp = lambda M, N, K: {"M": M, "N": N, "K": K, "ms": 1.0, "tops": 500.0,
                           "frac_of_bf16_peak": 0.25}
    line = {"clocks": {"sm_mhz": 2070.0},
            "prefill": {"shapes": [shp(2048, 12288, 4096), shp(2048, 4096, 12288)]},
            "prefill_long_context": {"shapes": [shp(18432, 17408, 5120), shp(18432, 5120, 17408)]},
            "moe": {"total": {"ms": 0.6, "frac_of_hbm": 0.14}, "gate_up": {"ms": 0.4},
                    "down": {"ms": 0.2}},
            "moe_layer": {"total_ms": 0.65, "frac_of_hbm_weights": 0.1},
            "decode_m4": {"gbs": 4600.0},
            "next_rows": {"kv3_encode": {"frac_of_hbm": 0.5, "frac_of_copy": 0.8}, "l2": "flushed"}}
    clk = {"sm_mhz": 2070.0, "samples": 12, "reasons": []}
    bench.flatten_sections(line, {"hbm_gbs": 6680.8},
                           {"prefill": clk, "longctx": clk, "moe": clk, "decode_m4": clk})
    for k in ("prefill_2048x12288x4096_tops", "prefill_2048x4096x12288_tops",
              "longctx_18432x17408x5120_tops", "longctx_18432x5120x17408_tops", "moe_total_ms",
              "prefill_sm_mhz", "moe_throttle", "decode_m4_frac", "next_kv3_encode_frac",
              "next_kv3_encode_frac_of_copy"):
        assert k in line and k in line["prefill"], k
        assert not isinstance(line[k], (list, dict))
    assert line["clocks"]["prefill_reasons"] == "none"
    json.dumps(line)
