"""GPU parity of the block-scaled expert path (moe_ffn_forward_mx) against the
fp64 oracle on the exactly dequantized weights.

Formats of DeepSeek-V4.1's official draft checkpoint (SpecForge PR #1073,
commit note on its export formats): FP4 routed experts (e2m1 codes, the even
input in the low nibble, one e8m0 scale per 32 inputs), FP8 linears (e4m3, one
e8m0 scale per 32 x 32 block) -- here the shared expert, and, as the other
routed-expert format, FP8 experts.  The tensor cores' block-scaled MMA takes
the codes and scales as they are; x and h enter as sums of e4m3 pieces.  Bars
as for the bf16 path: routing exact, largest output error within 2e-2 of the
output's RMS (or 1.25 x the bf16 rounding of the exact output where that
alone exceeds it), and at full size every output within one bf16 ulp of the
exact output.
"""
import numpy as np
import pytest
import torch

import oracle as O
from moe_ffn_speculative_gb300 import ops
from moe_ffn_speculative_gb300 import synthetic as S
from moe_ffn_speculative_gb300.build import build
from parity_util import (Y_TOL, beyond_one_ulp, compare_routing, expert_coverage, np64, oracle_recipe,
                         output_rounding_error, max_abs_over_rms, report)

pytestmark = pytest.mark.gpu

E2E_MARGIN_TOL = 1e-4
E2E_W_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _library():
    build()
    ops.lib()
    torch.cuda.init()


def _cfg(name, **kw):
    return S.LayerConfig(name, **kw)


SMALL = {
    # FP4 routed experts, one tile each, no shared expert (y written directly
    # at top-1; top-2 here goes through the combine)
    "fp4_tiny": _cfg("mx_fp4_tiny", T=16, H=128, E=8, I=128, K=2, expert_format="fp4", seed=61),
    # FP4 routed + FP8 shared expert with its sigmoid gate, router bias, two
    # gate_up tiles per expert, two output tiles
    "fp4_gated_fp8_shared": _cfg("mx_fp4_gated", T=37, H=512, E=8, I=256, K=2, shared_I=128, shared_gated=True,
                                 router_bias_std=0.1, expert_format="fp4", shared_format="fp8", seed=62),
    # the DeepSeek-V4 recipe on FP4 experts with the FP8 ungated shared expert
    "fp4_dsv4_recipe": _cfg("mx_fp4_dsv4", T=40, H=256, E=16, I=256, K=6, score_fn=S.SQRTSOFTPLUS,
                            expert_bias_std=0.05, route_scale=1.5, swiglu_limit=10.0, shared_I=256,
                            expert_format="fp4", shared_format="fp8", seed=63),
    # many tokens per expert: several 32-token tiles per expert
    "fp4_wide_tokens": _cfg("mx_fp4_wide", T=200, H=128, E=4, I=128, K=2, expert_format="fp4", seed=64),
    # FP8 routed experts (32 x 32 block scales) + FP8 shared expert
    "fp8_routed": _cfg("mx_fp8", T=24, H=256, E=8, I=384, K=2, shared_I=128, expert_format="fp8",
                       shared_format="fp8", seed=65),
    # top-1 FP8 experts without a shared expert: y written by the down epilogue
    "fp8_top1_direct": _cfg("mx_fp8_top1", T=72, H=256, E=8, I=256, K=1, expert_format="fp8", seed=66),
    # one token: one piece row group per token block, every other row zero
    "fp4_one_token": _cfg("mx_fp4_one", T=1, H=128, E=8, I=128, K=2, shared_I=128, expert_format="fp4",
                          shared_format="fp8", seed=70),
    # every expert selected by every token (K = E)
    "fp8_all_experts": _cfg("mx_fp8_all", T=30, H=128, E=4, I=128, K=4, expert_format="fp8", seed=69),
    # more than 1024 tokens: the router's logits GEMM, then select and permute
    "fp4_many_tokens": _cfg("mx_fp4_many", T=1100, H=128, E=12, I=128, K=2, shared_I=128, shared_gated=True,
                            expert_format="fp4", shared_format="fp8", seed=67),
}


def _cuda(d):
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


def _getter(cfg, d):
    """e -> the exactly dequantized (w_gate_up[e], w_down[e]), float64."""
    q, s = d["w_gate_up_q"].cpu().numpy(), d["w_gate_up_s"].cpu().numpy()
    dq, ds = d["w_down_q"].cpu().numpy(), d["w_down_s"].cpu().numpy()
    dec = O.dequant_fp4 if cfg.expert_format == "fp4" else O.dequant_fp8_blocks

    def get(e):
        return dec(q[e], s[e]), dec(dq[e], ds[e])
    return get


def _shared(cfg, d):
    if cfg.shared_I == 0:
        return None
    if cfg.shared_format == "fp8":
        return (O.dequant_fp8_blocks(d["sh_gate_up_q"].cpu().numpy(), d["sh_gate_up_s"].cpu().numpy()),
                O.dequant_fp8_blocks(d["sh_down_q"].cpu().numpy(), d["sh_down_s"].cpu().numpy()))
    return np64(d["sh_gate_up"]), np64(d["sh_down"])


def _oracle(cfg, d):
    orec = oracle_recipe(cfg)
    x64, gate64 = np64(d["x"]), np64(d["gate"])
    logits = O.router_logits(x64, gate64, np64(d["router_bias"]))
    _, oidx, ow, c = O.route_from_logits(logits, orec, np64(d["expert_bias"]))
    margin = O.selection_margin(c, oidx, orec)
    y = O.moe_combine_rows(x64, oidx, ow, _getter(cfg, d), cfg.swiglu_limit, _shared(cfg, d), np64(d.get("sh_gate")))
    return oidx, ow, margin, y


def _run(cfg, d):
    layer = ops.MoELayer(d, ops.Recipe.from_config(cfg), cfg.T, mx=True)
    assert layer.mx
    idx = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    y = layer.forward(d["x"], topk_idx_out=idx, topk_w_out=w, counts_out=counts)
    torch.cuda.synchronize()
    return layer, y, idx, w, counts


def _check(cfg, d, name, full):
    layer, y, idx, w, counts = _run(cfg, d)
    assert layer.ws.device_status() == (0, 0)
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
    report(test="mx_layer_full" if full else "mx_layer_small", case=name, max_abs_over_rms=err,
           output_rounding=out_round, tol=tol, beyond_one_ulp=n_ulp, rows=cfg.T, experts_covered=reached,
           experts_touched=touched)
    assert reached == touched
    assert err <= tol, f"max |dy| / RMS(y) = {err} (bf16 output rounding alone {out_round})"
    if full:
        assert n_ulp == 0, f"{n_ulp} outputs farther than one bf16 ulp from the exact output"
    y2 = layer.forward(d["x"])
    torch.cuda.synchronize()
    assert torch.equal(y, y2), "not deterministic"
    assert layer.ws.device_status() == (0, 0)


@pytest.mark.parametrize("name", list(SMALL))
def test_mx_layer_small(name):
    cfg = SMALL[name]
    _check(cfg, _cuda(S.make_inputs(cfg)), name, full=False)


# DeepSeek-V4.1's own draft layer in its checkpoint's formats (FP4 routed
# experts, FP8 shared expert); the V4-Flash drafter's shape with FP8 experts;
# the DeepSeek-V4-style layer with FP4 experts at 576 tokens (every expert
# touched, several token tiles per expert)
FULL = [("dsv41_dspark_draft", 72, "fp4"), ("dsv4_flash_drafter", 72, "fp8"), ("dsv4_style", 576, "fp4")]


@pytest.mark.parametrize("name,T,fmt", FULL)
def test_mx_layer_full_size(name, T, fmt):
    cfg = S.CONFIGS[name].with_(T=T, expert_format=fmt, shared_format="fp8")
    _check(cfg, S.make_inputs(cfg, device="cuda"), f"{name}_T{T}_{fmt}", full=True)


def test_mx_scale_chunks():
    """The prepared scales hold, for every (expert, tile, k-block), each
    128-row half's scales of its four 32-input chunks at byte
    16*(r%32) + 4*(r/32) + j of a 512-byte chunk (FP4: one scale per row;
    FP8: the 32 x 32 block's)."""
    for fmt in ("fp4", "fp8"):
        cfg = _cfg("mx_chunks", T=4, H=256, E=2, I=256, K=1, shared_I=128, expert_format=fmt, shared_format="fp8",
                   seed=68)
        d = _cuda(S.make_inputs(cfg))
        sc = ops.mx_prepare_scales(d).cpu().numpy()
        gs = d["w_gate_up_s"].cpu().numpy()
        E, H, I = cfg.E, cfg.H, cfg.I
        kb0 = H // 128
        for e in range(E):
            for m in range(I // 128):
                for kb in range(kb0):
                    blk = sc[((e * (I // 128) + m) * kb0 + kb) * 1024:][:1024]
                    for h in range(2):
                        for r in range(128):
                            row = h * I + m * 128 + r
                            for j in range(4):
                                want = gs[e, row, kb * 4 + j] if fmt == "fp4" else gs[e, row // 32, kb * 4 + j]
                                assert blk[h * 512 + 16 * (r % 32) + 4 * (r // 32) + j] == want


def test_mx_cuda_graph_replay():
    cfg = SMALL["fp4_gated_fp8_shared"]
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


def test_mx_refuses_unsupported_shapes():
    cfg = SMALL["fp4_tiny"]
    d = _cuda(S.make_inputs(cfg))
    rec = ops.Recipe.from_config(cfg)
    ws = ops.Workspace(ops.ffn_workspace_bytes(cfg.T, cfg.H, cfg.I, 0, rec))
    sc = ops.mx_prepare_scales(d)
    # H not a multiple of 128
    x = torch.zeros((cfg.T, 192), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((cfg.E, 192), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.MoeError) as e:
        ops.moe_ffn_forward_mx(x, g, ops.FMT_FP4, d["w_gate_up_q"], d["w_down_q"], sc, rec, ws, cfg.I)
    assert e.value.status == ops.MOE_ERR_UNSUPPORTED
    # scales too small
    with pytest.raises(ops.MoeError) as e:
        ops.moe_ffn_forward_mx(d["x"], d["gate"], ops.FMT_FP4, d["w_gate_up_q"], d["w_down_q"], sc[:1024], rec, ws,
                               cfg.I)
    assert e.value.status == ops.MOE_ERR_INVALID_ARG
    # an unknown format
    with pytest.raises(ops.MoeError) as e:
        ops.moe_ffn_forward_mx(d["x"], d["gate"], 7, d["w_gate_up_q"], d["w_down_q"], sc, rec, ws, cfg.I)
    assert e.value.status == ops.MOE_ERR_INVALID_ARG
