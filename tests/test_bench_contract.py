"""bench.py on the host: the algorithmic bytes and FLOPs it divides by, the
metric names of both arms, and the JSON line of the reference arm (the fp64
oracle on the host cores), which runs without a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from moe_ffn_speculative_gb300 import synthetic as S  # noqa: E402


# Per-layer bytes and FLOPs of the four decode workloads at their expected
# touched-expert counts U = E·(1 − (1 − K/E)^T) (fractional there, rounded
# here), tabulated independently of bench.py; bytes to three or four
# significant digits, FLOPs to two or three.
TABLE = [
    ("qwen3_8b_dspark", 8, 303e6, 2.7e9),
    ("qwen38_27b_dspark", 388, 6.18e9, 16.2e9),
    ("dsv3_style", 230, 20.35e9, 57.3e9),
    ("dsv4_style", 210, 5.30e9, 12.8e9),
]


@pytest.mark.parametrize("name,U,bytes_,flops", TABLE)
def test_algorithmic_bytes_and_flops_match_the_table(name, U, bytes_, flops):
    layer_bytes, ex_bytes, fl = bench.algorithmic(S.CONFIGS[name], U)
    assert abs(layer_bytes / bytes_ - 1) < 5e-3
    assert abs(fl / flops - 1) < 2e-2
    # the expert launch reads every touched weight once (and more: x, h, outputs)
    cfg = S.CONFIGS[name]
    weights = U * 3 * cfg.I * cfg.H * 2 + 3 * cfg.shared_I * cfg.H * 2
    assert ex_bytes > weights


def test_fp4_weights_count_half_a_byte_and_a_scale_per_32():
    cfg = S.CONFIGS["dsv41_dspark_draft"]
    b16, _, _ = bench.algorithmic(cfg, 100)
    b4, _, _ = bench.algorithmic(cfg.with_(expert_format="fp4"), 100)
    routed16 = 100 * 3 * cfg.I * cfg.H * 2
    assert b16 - b4 == pytest.approx(routed16 * (1 - (0.5 + 1 / 32) / 2), rel=1e-6)


def test_metric_names():
    assert bench.metric_for(S.CONFIGS["qwen3_8b_dspark"]) == bench.METRIC
    assert bench.metric_for(S.CONFIGS["dsv4_style"].with_(T=576)) == "MoE-FFN layer tokens/s (dsv4_style, T=576)"
    assert "FP4 experts" in bench.metric_for(S.CONFIGS["qwen3_8b_dspark"].with_(expert_format="fp4"))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 1
    assert line["value"] > 0 and line["config"]["workload"] == "qwen3_8b_dspark"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_under_torchrun_prints_one_line():
    """Two ranks (gloo on the host): rank 0 alone runs the oracle and prints
    the line; the other rank exits 0 without output."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


@pytest.mark.parametrize("name", ["qwen38_27b_dspark", "dsv3_style", "dsv4_style"])
def test_router_only_inputs_are_the_layers_own(name):
    """bench.py --route-only draws x, the gate and the biases as the full
    layer draws them first: the router it times sees the layer's operands."""
    import torch
    cfg = S.CONFIGS[name].with_(T=5, E=16, I=32, H=64, shared_I=32 if S.CONFIGS[name].shared_I else 0)
    full, router = S.make_inputs(cfg), S.make_router_inputs(cfg)
    for k in ("x", "gate", "router_bias", "expert_bias"):
        assert (full[k] is None and router[k] is None) or torch.equal(full[k], router[k]), k


def test_fused_layer_reports_back_to_back_and_isolated_launch_times():
    """The fused schedule's layer is one launch: its kernel time is the timed
    region's time per launch (consecutive launches overlap), and the launch on
    its own -- event nodes around it, their measured overhead taken off -- is
    reported beside it; other schedules report the event-node time minus the
    overhead."""
    from types import SimpleNamespace
    cfg = S.CONFIGS["qwen3_8b_dspark"]
    ev = {"event_pair_us": 5.0, "empty_launch_period_us": 1.1, "overhead_us": 3.9}
    wl = SimpleNamespace(cfg=cfg, sched="slice", ex_key="fused")
    roof, layer = bench.roofline_record(wl, 8, {"fused": 57.9}, 0.0499, 6780.0, 1942.5, "measured",
                                        "qwen3_8b_dspark", ev)
    assert roof["kernel_us"] == pytest.approx(49.9)
    assert roof["kernel_us_isolated"] == pytest.approx(54.0)
    assert roof["frac"] == pytest.approx(roof["algorithmic_bytes_per_launch"] / 49.9e-6 / 1e9 / 6780.0)
    assert roof["frac_isolated"] == pytest.approx(roof["algorithmic_bytes_per_launch"] / 54.0e-6 / 1e9 / 6780.0)
    assert layer["frac"] == pytest.approx(layer["roofline_us"] / 49.9)
    cfg4 = S.CONFIGS["dsv4_style"]
    wl4 = SimpleNamespace(cfg=cfg4, sched="stream_k", ex_key="experts")
    roof4, _ = bench.roofline_record(wl4, 210, {"router": 30.0, "experts": 752.0, "combine": 7.5}, 0.78, 6780.0,
                                     1942.5, "measured", "dsv4_style", ev)
    assert roof4["kernel_us"] == pytest.approx(748.1)
    assert "kernel_us_isolated" not in roof4
