"""The bench's reference arm on the host: it times the fp64 oracle on a bounded sample with one process per core
and prints the contract's JSON line (no GPU needed)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--config", "chain3_27b_bf16", "--cpu-workers", "2"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["unit"] == "nodes/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["n_gpus"] == 1
    assert line["steps"] == 2  # the passes actually timed
    assert line["config"]["workload"] == "chain3_27b_bf16"
    ex = line["extrapolation"]
    assert ex["attn_factor"] > 1 and ex["lm_factor"] > 1 and ex["round_s"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == line["value"] and cb["sample"]
    assert cb["nproc"] >= 1 and cb["cpu_model"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_default_workload_is_the_largest_single_gpu_config():
    sys.path.insert(0, ROOT)
    import bench
    from synth import configs

    assert bench.DEFAULT_CONFIG == "eagle64x32_27b_i8"
    big = max(configs.CONFIGS, key=lambda c: c.algorithmic_bytes())
    assert big.name == bench.DEFAULT_CONFIG
    assert bench.tensor_bound(configs.workload("eagle64x32_27b_i8"))
    assert not bench.tensor_bound(configs.workload("eagle32x8_27b_f16"))
    assert not bench.tensor_bound(configs.workload("specinfer16_27b_i8"))


def test_sliding_layers_keep_the_attention_intensity():
    # A sliding-window layer reads window + T - 1 positions and each row multiplies at most window keys, so its flop
    # per KV byte stays near a full layer's; the 32-node hybrid stays bound by HBM, as the full workload is.
    sys.path.insert(0, ROOT)
    import bench
    from synth import configs

    full = configs.workload("eagle32x8_27b_f16")
    intensity = lambda c: c.attention_flops() / (c.kv_bytes() + c.kv_scale_bytes())
    every_layer = configs.with_sliding_layers(full, 1024, full.n_layers + 1)
    assert all(every_layer.layer_window(l) == 1024 for l in range(full.n_layers))
    assert 0.95 < intensity(every_layer) / intensity(full) <= 1.0
    assert every_layer.attention_flops() < full.attention_flops() * 1024 / full.S
    assert not bench.tensor_bound(configs.with_sliding_layers(full, 1024, 6))
    assert bench.tensor_bound(configs.with_sliding_layers(configs.workload("eagle64x32_27b_i8"), 4096, 4))


def test_percentiles():
    sys.path.insert(0, ROOT)
    import bench

    xs = list(range(11))
    assert bench.pct(xs, 10) == 1 and bench.pct(xs, 50) == 5 and bench.pct(xs, 90) == 9
