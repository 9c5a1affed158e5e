"""The reference arm of the benchmark (the CPU oracle timed on the host
cores) prints one JSON line with the fields the measurement contract asks
for; run here on the tiny workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_bf16", "--steps", "3", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 3 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "one oracle call per step" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_both_arms_print_the_same_config_dict():
    """Both arms of bench.py describe the same workload with the same `config`
    object, built by one function, so a comparison of the two lines can match
    them."""
    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_layer_align_gb300 import inputs
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_bf16", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    d = json.loads([l for l in r.stdout.splitlines() if l.strip().startswith("{")][0])
    cfg = inputs.workload("tiny_bf16")
    assert d["config"] == bench.workload_config("tiny_bf16", cfg, list(cfg["T"]))
    assert d["config"]["workload"] == "tiny_bf16"


def test_roofline_fraction_picks_the_binding_limit():
    sys.path.insert(0, ROOT)
    import bench
    # 1 GB at 1000 GB/s = 1 ms; 1 TFLOP at 2000 TFLOP/s = 0.5 ms: HBM binds
    bound, frac, hbm, tc = bench.roofline_fractions(2000.0, 1e9, 1e12, 1000.0, 2000.0)
    assert bound == "hbm" and abs(frac - 0.5) < 1e-12 and abs(hbm - 0.5) < 1e-12
    assert abs(tc - 0.25) < 1e-12
    bound, frac, hbm, tc = bench.roofline_fractions(2000.0, 1e8, 4e12, 1000.0, 2000.0)
    assert bound == "tensor" and abs(frac - 1.0) < 1e-12
    # the layer's algorithmic work: touched experts' weights + logits + x + out
    nbytes, flops = bench.layer_work(2, 1, 4096, 14336, 8, 2, True)
    assert nbytes == 2 * 3 * 4096 * 14336 + 8 * 8 + 8 * 4 + 2 * 4096 * 2
    assert flops == 6.0 * 2 * 4096 * 14336


def test_weight_copies_keep_calls_out_of_l2():
    sys.path.insert(0, ROOT)
    import bench
    import torch
    from mixture_experts_layer_align_gb300 import inputs
    w = inputs.Weights(torch.zeros(2, 4), torch.zeros(2, 4), None, None, "bf16", 4, 2, 2)
    # 37.7 MB touched per call: 2 x 129 MiB / 37.7 MB -> 8 copies
    c = bench.weight_copies(w, 37_748_736, inputs)
    assert len(c) == -(-2 * bench.L2_BYTES // 37_748_736) and len(c) >= 7
    assert all(ci.w13.data_ptr() != w.w13.data_ptr() for ci in c[1:])
    assert len(bench.weight_copies(w, 10 ** 9, inputs)) == 2
