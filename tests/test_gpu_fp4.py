"""GPU parity of the FP4 routed-expert path (moe_ffn_forward_fp4) against the
fp64 oracle on the exactly dequantized weights.

The format is DeepSeek-V4.1's official one (SpecForge PR #1073, commit note on
the checkpoint's export formats): e2m1 codes, two per byte along the input
with the even input in the low nibble, one e8m0 scale per 32 inputs.  The
kernels expand the codes to f16 exactly and multiply x (as f16) by them with
fp32 accumulation, so the bars are those of the bf16 path: routing exact,
largest output error within 2e-2 of the output's RMS (or 1.25x the bf16
output rounding alone where that rounding exceeds it), and at full size every
output within one bf16 ulp of the exact output.
"""
import numpy as np
import pytest
import torch

import oracle as O
from moe_ffn_speculative_gb300 import ops
from moe_ffn_speculative_gb300 import synthetic as S
from moe_ffn_speculative_gb300.build import build
from parity_util import (Y_TOL, beyond_one_ulp, compare_routing, expert_coverage, np64, oracle_recipe,
                         output_rounding_error,
                         max_abs_over_rms, report)

pytestmark = pytest.mark.gpu

E2E_MARGIN_TOL = 1e-4
E2E_W_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _library():
    build()
    ops.lib()
    torch.cuda.init()


F = "fp4"
SMALL = {
    # one tile per expert, 16 tokens
    "fp4_tiny": S.LayerConfig("fp4_tiny", T=16, H=128, E=8, I=128, K=2, expert_format=F, seed=31),
    # ragged gate_up tile (I = 192), ragged down tile (H = 320), ragged
    # bf16 shared expert (Is = 200) with its sigmoid gate, router bias
    "fp4_ragged_gated_shared": S.LayerConfig("fp4_ragged_gated_shared", T=37, H=320, E=8, I=192, K=2,
                                             shared_I=200, shared_gated=True, router_bias_std=0.1,
                                             expert_format=F, seed=32),
    # the DeepSeek-V4 recipe: sqrt(softplus), selection bias, scale, clamp,
    # ungated shared expert
    "fp4_dsv4_recipe": S.LayerConfig("fp4_dsv4_recipe", T=40, H=256, E=16, I=256, K=6,
                                     score_fn=S.SQRTSOFTPLUS, expert_bias_std=0.05, route_scale=1.5,
                                     swiglu_limit=10.0, shared_I=256, expert_format=F, seed=33),
    # many tokens per expert: wide token tiles (n_max = 208)
    "fp4_wide_tokens": S.LayerConfig("fp4_wide_tokens", T=200, H=128, E=4, I=128, K=2, expert_format=F,
                                     seed=34),
}


def _cuda(d):
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


def _getter(d):
    """e -> the exactly dequantized (w_gate_up[e], w_down[e]), float64."""
    q, s = d["w_gate_up_q"].cpu().numpy(), d["w_gate_up_s"].cpu().numpy()
    dq, ds = d["w_down_q"].cpu().numpy(), d["w_down_s"].cpu().numpy()

    def get(e):
        return O.dequant_fp4(q[e], s[e]), O.dequant_fp4(dq[e], ds[e])
    return get


def _oracle(cfg, d, rows=None):
    orec = oracle_recipe(cfg)
    x64, gate64 = np64(d["x"]), np64(d["gate"])
    logits = O.router_logits(x64, gate64, np64(d["router_bias"]))
    _, oidx, ow, c = O.route_from_logits(logits, orec, np64(d["expert_bias"]))
    margin = O.selection_margin(c, oidx, orec)
    rows = np.arange(cfg.T) if rows is None else rows
    shared = None if d.get("sh_gate_up") is None else (np64(d["sh_gate_up"]), np64(d["sh_down"]))
    y = O.moe_combine_rows(x64[rows], oidx[rows], ow[rows], _getter(d), cfg.swiglu_limit, shared,
                           np64(d.get("sh_gate")))
    return oidx, ow, margin, y


def _run(cfg, d):
    layer = ops.MoELayer(d, ops.Recipe.from_config(cfg), cfg.T, mx=False)
    assert layer.fp4
    idx = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    y = layer.forward(d["x"], topk_idx_out=idx, topk_w_out=w, counts_out=counts)
    torch.cuda.synchronize()
    return layer, y, idx, w, counts


@pytest.mark.parametrize("name", list(SMALL))
def test_fp4_layer_small(name):
    cfg = SMALL[name]
    d = _cuda(S.make_inputs(cfg))
    layer, y, idx, w, counts = _run(cfg, d)
    oidx, ow, margin, y_ref = _oracle(cfg, d)
    n_amb, _ = compare_routing(idx, w, oidx, ow, margin, w_tol=E2E_W_TOL, margin_tol=E2E_MARGIN_TOL)
    assert n_amb == 0
    np.testing.assert_array_equal(counts.cpu().numpy(), np.bincount(oidx.reshape(-1), minlength=cfg.E))
    err = max_abs_over_rms(y, y_ref)
    out_round = output_rounding_error(y_ref)
    tol = max(Y_TOL, 1.25 * out_round)
    report(test="fp4_layer_small", case=name, max_abs_over_rms=err, output_rounding=out_round, tol=tol)
    assert err <= tol, f"max |dy| / RMS(y) = {err} (bf16 output rounding alone {out_round})"
    assert layer.ws.device_status() == (0, 0)
    y2 = layer.forward(d["x"])
    torch.cuda.synchronize()
    assert torch.equal(y, y2), "not deterministic"


FULL = [("dsv41_dspark_draft", 72), ("dsv4_flash_drafter", 72), ("dsv4_style", 576)]


@pytest.mark.parametrize("name,T", FULL)
def test_fp4_layer_full_size(name, T):
    """Every output row against the oracle, so every touched expert's FP4
    tiles meet it."""
    cfg = S.CONFIGS[name].with_(T=T, expert_format=F)
    d = S.make_inputs(cfg, device="cuda")
    layer, y, idx, w, counts = _run(cfg, d)
    oidx, ow, margin, y_ref = _oracle(cfg, d)
    n_amb, _ = compare_routing(idx, w, oidx, ow, margin, w_tol=E2E_W_TOL, margin_tol=E2E_MARGIN_TOL)
    assert n_amb == 0
    gcounts = counts.cpu().numpy()
    np.testing.assert_array_equal(gcounts, np.bincount(oidx.reshape(-1), minlength=cfg.E))
    reached, touched = expert_coverage(oidx, gcounts)
    err = max_abs_over_rms(y, y_ref)
    out_round = output_rounding_error(y_ref)
    tol = max(Y_TOL, 1.25 * out_round)
    n_ulp = beyond_one_ulp(y, y_ref)
    report(test="fp4_layer_full", case=f"{name}_T{T}", max_abs_over_rms=err, output_rounding=out_round, tol=tol,
           beyond_one_ulp=n_ulp, rows=T, experts_covered=reached, experts_touched=touched)
    assert reached == touched
    assert err <= tol, f"max |dy| / RMS(y) = {err} (bf16 output rounding alone: {out_round})"
    assert n_ulp == 0, f"{n_ulp} outputs farther than one bf16 ulp from the exact output"
    assert layer.ws.device_status() == (0, 0)


def test_fp4_scale_layout_round_trip():
    """The re-laid scales hold, for every (expert, tile, k-block), the scale
    pairs of its two 128-row halves; rows past the matrix hold scale 1."""
    cfg = SMALL["fp4_ragged_gated_shared"]
    d = _cuda(S.make_inputs(cfg))
    sc = ops.fp4_prepare_scales(d["w_gate_up_s"], d["w_down_s"]).cpu().numpy()
    gs, ds = d["w_gate_up_s"].cpu().numpy(), d["w_down_s"].cpu().numpy()
    E, H, I = cfg.E, cfg.H, cfg.I
    mb0, kb0, mb1, kb1 = -(-I // 128), H // 64, -(-H // 256), I // 64
    a = sc[:E * mb0 * kb0 * 512].reshape(E, mb0, kb0, 2, 128, 2)
    b = sc[E * mb0 * kb0 * 512:].reshape(E, mb1, kb1, 2, 128, 2)
    for e in range(E):
        for m in range(mb0):
            for h in range(2):
                for r in range(128):
                    row = m * 128 + r
                    want = gs[e, h * I + row].reshape(kb0, 2) if row < I else np.full((kb0, 2), 127)
                    np.testing.assert_array_equal(a[e, m, :, h, r], want)
        for m in range(mb1):
            for h in range(2):
                for r in range(128):
                    row = m * 256 + h * 128 + r
                    want = ds[e, row].reshape(kb1, 2) if row < H else np.full((kb1, 2), 127)
                    np.testing.assert_array_equal(b[e, m, :, h, r], want)


def test_fp4_cuda_graph_replay():
    cfg = SMALL["fp4_ragged_gated_shared"]
    d = _cuda(S.make_inputs(cfg))
    layer, y_ref, *_ = _run(cfg, d)
    s = torch.cuda.Stream()
    y = torch.empty_like(y_ref)
    with torch.cuda.stream(s):
        layer.forward(d["x"], y=y, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(d["x"], y=y, stream=s)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
    assert layer.ws.device_status() == (0, 0)


def test_fp4_scale_outside_exact_range_is_reported():
    """A block scale outside [104, 140] (products no longer exact in f16) is
    reported as MOE_ERR_DEVICE_RANGE; the forward still completes."""
    cfg = SMALL["fp4_tiny"]
    d = _cuda(S.make_inputs(cfg))
    layer, *_ = _run(cfg, d)
    assert layer.ws.device_status() == (0, 0)
    d2 = dict(d)
    d2["w_gate_up_s"] = d["w_gate_up_s"].clone()
    d2["w_gate_up_s"][:, 0, 0] = 150  # row 0 of every expert: touched by any routing
    layer2, *_ = _run(cfg, d2)
    assert layer2.ws.device_status() == (ops.MOE_ERR_DEVICE_RANGE, 12)
    assert layer2.ws.device_status() == (0, 0)  # read and cleared


def test_fp4_activation_outside_f16_range_is_reported():
    cfg = SMALL["fp4_tiny"]
    d = _cuda(S.make_inputs(cfg))
    d["x"][3, 5] = 1.0e5
    layer, *_ = _run(cfg, d)
    assert layer.ws.device_status() == (ops.MOE_ERR_DEVICE_RANGE, 13)


def test_fp4_refuses_unsupported_shapes():
    cfg = SMALL["fp4_tiny"]
    d = _cuda(S.make_inputs(cfg))
    rec = ops.Recipe.from_config(cfg)
    ws = ops.Workspace(ops.ffn_workspace_bytes(cfg.T, cfg.H, cfg.I, 0, rec))
    sc = ops.fp4_prepare_scales(d["w_gate_up_s"], d["w_down_s"])
    # H not a multiple of 64
    x = torch.zeros((cfg.T, 96), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((cfg.E, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.MoeError) as e:
        ops.moe_ffn_forward_fp4(x, g, d["w_gate_up_q"], d["w_down_q"], sc, rec, ws)
    assert e.value.status == ops.MOE_ERR_UNSUPPORTED
    # scales buffer too small
    with pytest.raises(ops.MoeError) as e:
        ops.moe_ffn_forward_fp4(d["x"], d["gate"], d["w_gate_up_q"], d["w_down_q"], sc[:256], rec, ws)
    assert e.value.status == ops.MOE_ERR_INVALID_ARG
