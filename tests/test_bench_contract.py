"""The JSON line of bench.py: the keys, types and cross-arm consistency that the benchmark
contract asks for (one line on stdout; the reference arm times the oracle and runs on CPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e")


def _bench(*args, timeout=900):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


def _check_base(line, steps, warmup):
    for k in BASE_KEYS:
        assert k in line, k
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["steps"] == steps and line["warmup"] == warmup and line["n_gpus"] == 1
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["config"]["workload"] and line["config"]["global_batch"] == line["config"]["T"]
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == line["unit"]
    assert "h2d_bytes_per_step" in e2e and "d2h_bytes_per_step" in e2e


def test_reference_arm_line():
    line = _bench("--impl", "reference", "--config", "tiny_f32", "--steps", "2", "--warmup", "3")
    _check_base(line, 2, 3)
    assert line["impl"] == "reference"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert cb["unit"] == line["unit"] and cb["sample"]
    assert line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_line_matches_the_reference_arm():
    ours = _bench("--config", "2b_bf16", "--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    _check_base(ours, 3, 3)
    roof = ours["roofline"]
    assert roof["bound"] in ("tensor", "hbm") and roof["unit"] in ("TFLOP/s", "GB/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert "traffic" in roof
    assert ours["gpu_launches"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(ours["clocks"])
    assert ours["e2e"]["h2d_bytes_per_step"] > 0 and ours["e2e"]["d2h_bytes_per_step"] > 0
    ref = _bench("--impl", "reference", "--config", "2b_bf16", "--steps", "1", "--warmup", "3")
    for k in ("metric", "unit", "higher_is_better", "config"):
        assert ours[k] == ref[k], k


def test_roofline_inputs_of_the_routed_gate_up_launch():
    """The roofline describes one gate/up launch: over the routed groups only when the shared
    group has a launch of its own, over every group otherwise."""
    sys.path.insert(0, ROOT)
    import bench
    import moe_inputs
    sh = moe_inputs.CONFIGS["16b_bf16"]
    T = sh.T
    routed = 4.0 * sh.d * sh.inter * T * sh.top_k
    assert bench.gate_up_flops(sh, T, with_shared=False) == routed
    assert bench.gate_up_flops(sh, T) == routed * (sh.top_k + sh.n_shared) / sh.top_k
    every_expert = [1] * sh.n_routed
    # routed weights + permuted rows read, activations written (bf16)
    want = (sh.n_routed * 2 * sh.inter * sh.d + T * sh.top_k * sh.d + T * sh.top_k * sh.inter) * 2
    assert bench.gate_up_bytes(sh, T, every_expert, with_shared=False) == want
    assert bench.gate_up_traffic("16b_bf16", "gemm_gate_up_routed") == 1141014016 + 259321856
    assert bench.gate_up_traffic("2b_bf16", "gemm_gate_up_routed") is None


def test_layer_roofline_of_the_scope_table():
    """The layer roofline of the 16B-like prefill is its FLOPs at the bf16 peak (2.27 TFLOP), and
    that of the T = 64 decode its weight bytes at the HBM bandwidth (66 experts x 3 x 1408 x 2048
    bf16 = 1.142 GB when every routed expert receives a token)."""
    import bench
    sh = bench.moe_inputs.CONFIGS["16b_bf16"]
    r = bench.layer_roofline(sh, sh.T, [1] * sh.n_routed, 6500.0, 1800.0)
    assert r["bound"] == "tensor"
    assert abs(r["flops"] - 138.7e6 * sh.T) / r["flops"] < 1e-3
    assert abs(r["roofline_ms"] - r["flops"] / 1.8e15 * 1e3) < 1e-9
    dec = bench.moe_inputs.CONFIGS["16b_decode_bf16"]
    r = bench.layer_roofline(dec, dec.T, [1] * dec.n_routed, 6500.0, 1800.0)
    assert r["bound"] == "hbm"
    weights = 66 * 3 * 1408 * 2048 * 2
    assert weights < r["bytes"] < weights + 2e6
    assert abs(r["roofline_ms"] - 0.1757) < 0.001
    # untouched experts do not count
    r2 = bench.layer_roofline(dec, dec.T, [1] * 32 + [0] * 32, 6500.0, 1800.0)
    assert r2["bytes"] < r["bytes"] - 32 * 3 * 1408 * 2048 * 2 + 1
