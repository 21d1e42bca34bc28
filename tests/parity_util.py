"""Helpers shared by the GPU parity tests: convert inputs for the oracle,
compare routing with the ambiguity rule, measure output error."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from moe_ffn_speculative_gb300.synthetic import LayerConfig

# Output tolerance: max |y_gpu - y_oracle| / RMS(y_oracle) for bf16 weights,
# bf16 activations between the two GEMMs and fp32 accumulation.
Y_TOL = 2e-2
# Routing weights from identical fp32 logits.
W_ABS_TOL = 1e-6
# A selection made on fp32 shifted scores may differ from the fp64 one only
# where the oracle's deciding gap is below this (a few fp32 ulps of O(1) values).
MARGIN_TOL = 1e-5


def np64(t):
    return None if t is None else t.detach().to("cpu").to(torch.float64).numpy()


def oracle_recipe(cfg: LayerConfig, **over) -> O.Recipe:
    kw = dict(num_experts=cfg.E, top_k=cfg.K, score_fn=cfg.score_fn, n_group=cfg.n_group,
              topk_group=cfg.topk_group, group_topn=cfg.group_topn, norm_topk_prob=cfg.norm_topk_prob,
              norm_eps=cfg.norm_eps, route_scale=cfg.route_scale, swiglu_limit=cfg.swiglu_limit)
    kw.update(over)
    return O.Recipe(**kw)


def compare_routing(idx_gpu, w_gpu, o_idx, o_w, o_margin, w_tol=W_ABS_TOL, margin_tol=MARGIN_TOL):
    """Rows whose picks differ must be ambiguous (oracle margin < margin_tol);
    every other row must match exactly, with weights within w_tol.  Returns
    (number of ambiguous rows, boolean mask of the rows that match)."""
    ig = idx_gpu.cpu().numpy().astype(np.int64)
    wg = w_gpu.cpu().numpy().astype(np.float64)
    same = np.all(ig == o_idx, axis=1)
    bad = (~same) & (o_margin >= margin_tol)
    assert not bad.any(), (
        f"{bad.sum()} rows select different experts with a clear margin; first row "
        f"{np.nonzero(bad)[0][0]}: gpu {ig[bad][0]} oracle {o_idx[bad][0]} margin {o_margin[bad][0]}")
    if same.any():
        err = np.abs(wg[same] - o_w[same]).max()
        assert err <= w_tol, f"routing weight error {err} > {w_tol}"
    return int((~same).sum()), same


def max_abs_over_rms(y_gpu, y_ref) -> float:
    yg = y_gpu.detach().to("cpu").to(torch.float64).numpy()
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    return float(np.abs(yg - y_ref).max() / rms)


def expert_getter(d):
    """e -> (w_gate_up[e], w_down[e]) as float64 on the CPU, copied slice by slice."""
    def get(e):
        return np64(d["w_gate_up"][e]), np64(d["w_down"][e])
    return get


def oracle_rows(d, cfg: LayerConfig, rows, idx_rows, w_rows):
    """Oracle y for the given token rows with the given routing."""
    x = np64(d["x"][rows])
    shared = None
    if d.get("sh_gate_up") is not None:
        shared = (np64(d["sh_gate_up"]), np64(d["sh_down"]))
    return O.moe_combine_rows(x, idx_rows, w_rows, expert_getter(d), cfg.swiglu_limit, shared,
                              np64(d.get("sh_gate")))


def logits_bound(x64, gate64):
    """Bound on |fp32 logit - exact logit| for sums of H exact products
    accumulated in fp32: H * 2^-24 * sum_h |x_h g_h| (per token, expert)."""
    H = x64.shape[1]
    return H * 2.0 ** -24 * (np.abs(x64) @ np.abs(gate64).T)


def bf(a):
    """Round to bf16 (nearest even) and back to float64."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).to(torch.float64).numpy()


def bf_pair(a):
    """The compensated pair hi + lo of bf16 that carries h between the GEMMs."""
    hi = bf(a)
    return hi + bf(a - hi)


def beyond_one_ulp(y_gpu, y_ref, abs_floor_rms=1e-3) -> int:
    """Elements of the bf16 output farther from the exact output than one
    bf16 ulp of the exact value (plus abs_floor_rms x RMS, which covers the
    fp32 accumulation's absolute error on near-zero outputs).  An output that
    is the exact result rounded to bf16, give or take the last bit, has
    none."""
    yg = y_gpu.detach().to("cpu").to(torch.float64).numpy()
    _, ex = np.frexp(y_ref)
    ulp = np.ldexp(1.0, ex - 8)
    floor = abs_floor_rms * float(np.sqrt(np.mean(y_ref ** 2)))
    return int((np.abs(yg - y_ref) > ulp + floor).sum())


def output_rounding_error(y_ref):
    """max |dy| / RMS(y) of rounding the exact output to bf16 alone."""
    return float(np.abs(bf(y_ref) - y_ref).max() / np.sqrt(np.mean(y_ref ** 2)))


def expert_coverage(idx_rows, counts) -> tuple:
    """(touched experts that the compared rows reach, touched experts in the
    forward): the compared rows meet every expert tile the GPU streamed only
    when the two are equal."""
    touched = set(np.nonzero(np.asarray(counts) > 0)[0].tolist())
    reached = set(np.unique(np.asarray(idx_rows)).tolist()) & touched
    return len(reached), len(touched)


def report(**kw):
    """Append one parity record to $MOE_PARITY_REPORT (a JSON-lines file)."""
    import json
    import os
    path = os.environ.get("MOE_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(kw) + "\n")


def bf16_floor_error(d, cfg: LayerConfig, rows, idx_rows, w_rows, y_ref):
    """max |dy| / RMS(y) that the roundings the path prescribes -- h carried as a
    bf16 hi + lo pair between the GEMMs, the output y in bf16 -- produce on
    their own (everything else exact, fp64)."""

    x = np64(d["x"][rows])
    ye = np.zeros_like(y_ref)
    for e in np.unique(idx_rows):
        wgu, wd = np64(d["w_gate_up"][int(e)]), np64(d["w_down"][int(e)])
        rr, kk = np.nonzero(idx_rows == e)
        gu = x[rr] @ wgu.T
        i = wgu.shape[0] // 2
        h = bf_pair(O.swiglu(gu[:, :i], gu[:, i:], cfg.swiglu_limit))
        ye[rr] += w_rows[rr, kk][:, None] * (h @ wd.T)
    if d.get("sh_gate_up") is not None:
        sgu, sd = np64(d["sh_gate_up"]), np64(d["sh_down"])
        gu = x @ sgu.T
        i = sgu.shape[0] // 2
        hs = bf_pair(O.swiglu(gu[:, :i], gu[:, i:], cfg.swiglu_limit))
        ye += O.shared_gate(x, np64(d.get("sh_gate")))[:, None] * (hs @ sd.T)
    ye = bf(ye)
    return float(np.abs(ye - y_ref).max() / np.sqrt(np.mean(y_ref ** 2)))
