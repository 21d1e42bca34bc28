"""Benchmark of the MoE-FFN layer forward on GB300.

Default workload: the Qwen3-8B DSpark draft MoE layer at T=72 tokens (8
requests x verify block 9), H=4096, E=8 experts of I=1536, top-1 softmax,
renormalised; synthetic seeded inputs and random-init bf16 weights.

One step = one full layer forward (router, permutation, grouped gate_up,
grouped down, combine) through the library's C ABI, replayed from a CUDA
graph.  Weights rotate over several copies whose total exceeds the L2 cache,
so every step streams its weights from HBM.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead (the reference arm of this method: no other implementation
of it exists to run).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_ffn_speculative_gb300 import synthetic as S  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "MoE-FFN layer tokens/s at T=72 on 1 GB300"
UNIT = "tokens/s"


def metric_for(cfg) -> str:
    """The headline metric for the headline layer, else one naming the
    workload (both arms print the same name for the same workload)."""
    fp4 = cfg.expert_format == "fp4"
    if cfg.name == "qwen3_8b_dspark" and cfg.T == 72 and not fp4:
        return METRIC
    return f"MoE-FFN layer tokens/s ({cfg.name}{', FP4 experts' if fp4 else ''}, T={cfg.T})"


CSRC = os.path.join(ROOT, "moe_ffn_speculative_gb300", "csrc")
# per expert schedule: the dominant kernel, its ncu summary prefix, its source
KERNELS = {"stream_k": ("moe_experts_kernel", "experts_kernel", "gemm.cu"),
           "slice": ("moe_slice_kernel", "slice_kernel", "slice.cu")}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="qwen3_8b_dspark", choices=list(S.CONFIGS))
    ap.add_argument("--tokens", type=int, default=None, help="override T of the workload")
    ap.add_argument("--experts", type=int, default=None, help="override E (small profiling cases)")
    ap.add_argument("--schedule", default="auto", choices=["auto", "stream_k", "slice"],
                    help="expert schedule (auto: the library's choice for the shape)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "fp4"],
                    help="routed experts' format: bf16, or FP4 (e2m1 codes + e8m0 scale per 32 inputs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed

def dist_setup(n):
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- roofline helpers

def algorithmic(cfg, counts_u: int):
    """Bytes and FLOPs of one layer forward and of its expert-GEMM launch,
    counting only the touched experts' weights (each read once)."""
    T, H, I, E, K, Is = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.shared_I
    # routed weights: bf16, or FP4 codes (half a byte) plus one scale byte per 32
    wb = (0.5 + 1 / 32) if cfg.expert_format == "fp4" else 2
    gu_w = int(counts_u * 2 * I * H * wb) + 2 * Is * H * 2
    dn_w = int(counts_u * H * I * wb) + H * Is * 2
    act = T * H * 2 * 2  # x read, y written
    gate = E * H * 2 + (H * 2 if cfg.shared_gated else 0)
    biases = E * 4 * ((cfg.router_bias_std > 0) + (cfg.expert_bias_std > 0))
    layer_bytes = gu_w + dn_w + act + gate + biases
    rows = T * K + (T if Is else 0)
    # experts launch: both projections' weights once, x gathered, h (hi and lo)
    # written and read back, the weighted outputs written (fp32 rows, or bf16 y)
    out = rows * H * 4 if (K > 1 or Is) else T * H * 2
    ex_bytes = gu_w + dn_w + T * H * 2 + 2 * rows * max(I, Is) * 2 * 2 + out
    flops = T * K * 6 * H * I + (T * 6 * H * Is if Is else 0) + 2 * T * H * E
    return layer_bytes, ex_bytes, flops


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def ncu_traffic(schedule: str, workload: str):
    """Per-launch DRAM traffic of the schedule's dominant kernel from the
    committed ncu summary, or None when its source changed since the capture."""
    _, prefix, src = KERNELS[schedule]
    path = os.path.join(ROOT, "profiles", f"{prefix}_{workload}.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        text = f.read()
    m = re.search(r"traffic_bytes_per_launch\s*=\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256\s*=\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    with open(os.path.join(CSRC, src), "rb") as f:
        cur = hashlib.sha256(f.read()).hexdigest()
    return float(m.group(1)) if cur == h.group(1) else None


# ----------------------------------------------------------------------------- CPU oracle

def cpu_oracle_pass(cfg, host, w64, tokens):
    """The oracle on `tokens` rows of the workload: routing from exact logits,
    then the experts the rows select.  Expert weights come pre-converted."""
    import oracle as O
    x = host["x"][tokens].double().numpy()
    f64 = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    rec = O.Recipe(cfg.E, cfg.K, cfg.score_fn, cfg.n_group, cfg.topk_group, cfg.group_topn,
                   cfg.norm_topk_prob, cfg.norm_eps, cfg.route_scale, cfg.swiglu_limit)
    logits = O.router_logits(x, f64(host["gate"]), f64(host["router_bias"]))
    _, idx, w, _ = O.route_from_logits(logits, rec, f64(host["expert_bias"]))
    shared = None if host["sh_gate_up"] is None else (w64["sh_gate_up"], w64["sh_down"])
    return O.moe_combine_rows(x, idx, w, lambda e: w64[e], cfg.swiglu_limit, shared, f64(host["sh_gate"]))


def cpu_prepare(cfg):
    import oracle as O
    host = S.make_inputs(cfg, device="cpu")
    w64 = {}
    for e in range(cfg.E):
        if cfg.expert_format == "fp4":
            w64[e] = (O.dequant_fp4(host["w_gate_up_q"][e].numpy(), host["w_gate_up_s"][e].numpy()),
                      O.dequant_fp4(host["w_down_q"][e].numpy(), host["w_down_s"][e].numpy()))
        else:
            w64[e] = (host["w_gate_up"][e].double().numpy(), host["w_down"][e].double().numpy())
    if host["sh_gate_up"] is not None:
        w64["sh_gate_up"] = host["sh_gate_up"].double().numpy()
        w64["sh_down"] = host["sh_down"].double().numpy()
    return host, w64


def cpu_baseline(cfg, seconds: float):
    host, w64 = cpu_prepare(cfg)
    t0 = time.perf_counter()
    n_tok = 0
    passes = 0
    while True:
        cpu_oracle_pass(cfg, host, w64, np.arange(cfg.T))
        n_tok += cfg.T
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": n_tok / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{passes} full layer passes of T={cfg.T} tokens ({dt:.1f} s), fp64 numpy oracle, "
                      f"expert weights pre-converted to fp64"}


def run_reference(args, cfg, rank, world):
    """The fp64 CPU oracle as the reference arm."""
    if rank != 0:
        return
    K = args.steps if args.steps is not None else 20
    W = args.warmup if args.warmup is not None else 3
    host, w64 = cpu_prepare(cfg)
    # size each step's token sample so the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    cpu_oracle_pass(cfg, host, w64, np.arange(cfg.T))
    t_layer = time.perf_counter() - t0
    per_tok = t_layer / cfg.T
    tok_per_step = int(max(1, min(cfg.T, 120.0 / max(K + W, 1) / per_tok)))
    rng = np.random.default_rng(0)
    samples = [rng.choice(cfg.T, tok_per_step, replace=False) for _ in range(K + W)]
    for i in range(W):
        cpu_oracle_pass(cfg, host, w64, samples[i])
    t0 = time.perf_counter()
    for i in range(K):
        cpu_oracle_pass(cfg, host, w64, samples[W + i])
    dt = time.perf_counter() - t0
    value = K * tok_per_step / dt
    line = {"metric": metric_for(cfg), "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": K, "warmup": W,
            "ms_per_step": dt / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I, "K": cfg.K,
                       "shared_I": cfg.shared_I,
                       "routed_experts": "fp4 (e2m1 + e8m0/32)" if cfg.expert_format == "fp4" else "bf16",
                       "tokens_per_step_sample": tok_per_step},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{tok_per_step} of the {cfg.T} tokens per step, fp64 numpy oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args, cfg, rank, world):
    from moe_ffn_speculative_gb300 import ops
    from moe_ffn_speculative_gb300.build import build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    build()
    dev = torch.device("cuda", torch.cuda.current_device())
    K = args.steps if args.steps is not None else 20000
    W = max(3, args.warmup if args.warmup is not None else 50)
    rec = ops.Recipe.from_config(cfg)
    fp4 = cfg.expert_format == "fp4"
    ops.set_schedule({"auto": ops.SCHEDULE_AUTO, "stream_k": ops.SCHEDULE_STREAM_K,
                      "slice": ops.SCHEDULE_SLICE}[args.schedule])
    # FP4 routed experts always run the stream-K schedule
    sched = "stream_k" if fp4 else ops.SCHEDULE_NAMES[ops.ffn_schedule(
        cfg.T, cfg.H, cfg.I, cfg.shared_I, rec, gated=cfg.shared_gated and cfg.shared_I > 0)]
    base = S.make_inputs(cfg, device=dev, seed=cfg.seed + 1000 * rank)
    n_copies = max(2, -(-4 * L2_BYTES // (cfg.weight_bytes + 1)))
    wkeys = ["w_gate_up_q", "w_down_q"] if fp4 else ["w_gate_up", "w_down"]
    layers = [base]
    for c in range(1, n_copies):
        dd = dict(base)
        for k in wkeys + (["sh_gate_up", "sh_down"] if base["sh_gate_up"] is not None else []):
            dd[k] = base[k].clone()
        layers.append(dd)
    if fp4:
        sc = ops.fp4_prepare_scales(base["w_gate_up_s"], base["w_down_s"])
        for dd in layers:
            dd["scales"] = sc.clone()
    ws = ops.Workspace(ops.ffn_workspace_bytes(cfg.T, cfg.H, cfg.I, cfg.shared_I, rec), dev)
    x = base["x"]
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(dd, xx, yy, cnt=None):
        kw = dict(router_bias=dd["router_bias"], expert_bias=dd["expert_bias"], sh_gate_up=dd["sh_gate_up"],
                  sh_down=dd["sh_down"], sh_gate=dd["sh_gate"], y=yy, counts_out=cnt, stream=stream)
        if fp4:
            ops.moe_ffn_forward_fp4(xx, dd["gate"], dd["w_gate_up_q"], dd["w_down_q"], dd["scales"], rec, ws, **kw)
        else:
            ops.moe_ffn_forward(xx, dd["gate"], dd["w_gate_up"], dd["w_down"], rec, ws, **kw)

    def fwd(i, yy=y, cnt=None):
        call(layers[i % n_copies], x, yy, cnt)

    with torch.cuda.stream(stream):
        fwd(0, cnt=counts)
    torch.cuda.synchronize()
    u = int((counts > 0).sum().item())
    st, info = ws.device_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} ({info}) after the first forward")

    # One CUDA graph of G consecutive layers (weight copies in turn), as a
    # decode step's graph holds a model's layers back to back; G divides K,
    # so exactly K layers are timed.
    G = next((g for g in (8, 6, 4, 2) if K % g == 0 and g % n_copies == 0), 1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            fwd(i)
    torch.cuda.synchronize()
    for i in range(-(-W // G)):
        graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(K // G):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_total = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / K
    value = cfg.T * K * world / (ms_total / 1e3)

    # per-kernel durations (eager launches, events around every kernel)
    n_prof = min(K, 400)
    n_k = 3
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * n_k)] for _ in range(n_prof)]
    for row in evs:  # torch creates the CUDA event on its first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            ops.set_profile_events(evs[i])
            fwd(i)
    ops.set_profile_events(None)
    torch.cuda.synchronize()
    if sched == "slice":
        # one fused launch, recorded as the expert-GEMM pair
        launched, timed = 1, {"fused": 1}
    else:
        launched = 3 if (cfg.K > 1 or cfg.shared_I > 0) else 2
        if cfg.T > 1024:  # the router's logits by a separate GEMM launch
            launched += 1
        timed = {n: k for k, n in enumerate(["router", "experts", "combine"][:launched])}
    per_kernel = {n: float(np.mean([e[2 * k].elapsed_time(e[2 * k + 1]) for e in evs])) * 1e3  # us
                  for n, k in timed.items()}

    # end to end: pinned host x -> device, forward, device y -> pinned host, every step
    x_host = base["x"].cpu().pin_memory()
    y_host = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    n_e2e = min(K, 2000)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(n_e2e):
            x_dev.copy_(x_host, non_blocking=True)
            call(layers[i % n_copies], x_dev, y)
            y_host.copy_(y, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = cfg.T * n_e2e * world / (ms_e2e / 1e3)
    st, info = ws.device_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} ({info}) after the timed region")

    hbm, tflops, peak_src = measured_peaks()
    layer_bytes, ex_bytes, flops = algorithmic(cfg, u)
    if sched == "slice":
        # the fused launch is the whole layer: its algorithmic bytes are the layer's
        ex_bytes = layer_bytes
    if sched == "slice":
        # the step is this one launch: its average duration over the timed
        # graph region (inter-kernel gaps included) is the step time
        t_ex = ms_step * 1e-3
    else:
        t_ex = per_kernel["experts"] * 1e-6
    achieved = ex_bytes / t_ex / 1e9
    layer_gbs = layer_bytes / (ms_step * 1e-3) / 1e9
    roof_layer_us = max(layer_bytes / (hbm * 1e9), flops / (tflops * 1e12)) * 1e6
    wl = cfg.name if args.tokens is None and args.experts is None else f"{cfg.name}_T{cfg.T}_E{cfg.E}"
    traffic = ncu_traffic(sched, wl + ("_fp4" if fp4 else ""))

    if rank != 0:
        return
    line = {
        "metric": metric_for(cfg),
        "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms_step,
        "us_per_layer": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # the MMA operand type: FP4 experts are expanded to f16 on chip
        "dtype": "f16" if fp4 else "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I, "K": cfg.K,
                   "shared_I": cfg.shared_I, "touched_experts": u, "schedule": sched,
                   "routed_experts": "fp4 (e2m1 + e8m0/32)" if fp4 else "bf16",
                   "launch": f"cuda_graph_replay, {G} layer{'s' if G > 1 else ''} per graph",
                   "l2": f"weights rotate over {n_copies} copies ({n_copies * cfg.weight_bytes / 1e9:.2f} GB) > L2",
                   "parallelism": "replicas" if world > 1 else "single_gpu"},
        "roofline": {"bound": "hbm", "kernel": KERNELS[sched][0], "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": ex_bytes},
        "layer_roofline": {"bytes": layer_bytes, "flops": flops, "roofline_us": roof_layer_us,
                           "achieved_gbs": layer_gbs, "frac": roof_layer_us / (ms_step * 1e3)},
        "kernel_us": per_kernel,
        "gpu_launches": launched * K,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": cfg.T * cfg.H * 2,
                "d2h_bytes_per_step": cfg.T * cfg.H * 2, "steps": n_e2e, "launch": "eager"},
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    cfg = S.CONFIGS[args.config]
    if args.weights == "fp4":
        cfg = cfg.with_(expert_format="fp4")
    if args.tokens is not None:
        cfg = cfg.with_(T=args.tokens)
    if args.experts is not None:
        cfg = cfg.with_(E=args.experts)
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, cfg, rank, world)
    else:
        run_gpu(args, cfg, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
