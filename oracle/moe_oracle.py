"""fp64 CPU oracle of the MoE-FFN layer forward of DFlash/DSpark draft models.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library.

Every step is written as the plain definition the pages give, in float64, on the
exact values of the bf16 / fp32 inputs (the caller converts them to float64).
Library primitives used as single steps: ``numpy`` matrix products, ``argmax``,
``argsort`` and ``bincount``.  No blocking, fusion or reordering beyond what the
definitions state.

Sources (web pages, cited by title and section):

* [P1] sglang PR #48763 "[Feat] dflash: Serve MoE FFN drafts for DFlash and
  DSpark" -- commit notes on DraftMoE forward (fp32 router logits, the
  sigmoid-gated shared expert added to the routed output, the empty-input rule)
  and on the three CUDA fixes (expert bias, routed_scaling_factor, shared expert
  read before the in-place experts).
* [P2] SpecForge PR #1033 "MoE FFN for DFlash-family drafts: the module" --
  section "Router" (the score -> select -> routing_weights table) and the commit
  note on the 1e-20 renormalisation epsilon.
* [P3] SpecForge PR #941 "SGLang draft classes for the Qwen3.8-27B DSpark MoE
  drafter ..." -- section "What" (fp32 logits with the folded centering bias,
  sigmoid-gated shared expert) and the follow-up comment on DeepSeek-V4 drafters
  (sqrtsoftplus, selection-only bias, groups, scaling, clamped SwiGLU, ungated
  shared expert with the same clamp).
* [P4] SpecForge PR #1073 "MoE drafts: DeepSeek-V4.1's own DSpark draft" --
  commit notes on the expert bias (it moves which experts are picked, not
  their weights), on select receiving the shifted scores, on the DeepSeek-V4 family (sqrt(softplus)
  scores, always renormalised, route_scale, clamped SwiGLU, one ungated shared
  expert), on the fused gate_up_proj / down_proj expert layout and on the
  export formats of the official checkpoint (FP4 routed experts, FP8 linears
  with 32 x 32 block scales).
* [P5] MoE-Infinity PR #143 "converge DFlash spec-decode stack" -- commit note
  on the resident GPT-OSS loader (MXFP4 codes and scales, uint8,
  output-major).

Readings of points the pages leave open:

* gate/up order inside ``gate_up_proj``: rows [0, I) are the gate (w1), rows
  [I, 2I) the up projection (w3).
* clamped SwiGLU with limit L > 0: gate clamped from above at L, up clamped to
  [-L, L], then silu(gate) * up.  The same limit applies to the shared expert.
* group score of group-limited select: the sum of the ``group_topn`` (=2)
  largest shifted scores in the group; groups outside the ``topk_group`` best
  are not selectable.
* ties: the lower expert (or group) index wins; the output order is descending
  shifted score.
* ``route_scale`` multiplies the routed weights only, never the shared expert.
* shared gate: one scalar per token, sigmoid(x_t . g) with g of shape [H].
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional, Tuple

import numpy as np

SCORE_SOFTMAX = 0
SCORE_SIGMOID = 1
SCORE_SQRTSOFTPLUS = 2


@dataclass(frozen=True)
class Recipe:
    """The routing recipe; the fields map the configuration keys the pages
    name (num_experts, num_experts_per_tok, scoring_func, n_group / topk_group,
    norm_topk_prob, routed_scaling_factor, swiglu_limit)."""

    num_experts: int
    top_k: int
    score_fn: int = SCORE_SOFTMAX
    n_group: int = 1
    topk_group: int = 1
    group_topn: int = 2
    norm_topk_prob: bool = True
    norm_eps: float = 1e-20
    route_scale: float = 1.0
    swiglu_limit: float = 0.0


# --------------------------------------------------------------------------
# Router, step "score" ([P2] Router table; [P1], [P3] fp32 logits with the
# folded bias; [P4] DeepSeek-V4 sqrt(softplus))
# --------------------------------------------------------------------------

def router_logits(x: np.ndarray, gate: np.ndarray,
                  router_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * gate[e, h] (+ router_bias[e]).

    The linear gate of the Router table ([P2] "score": weight [E, H]); the
    folded centering bias of [P3] "What" is added to the logits, so it moves
    both the selection and the weights."""
    logits = np.asarray(x, np.float64) @ np.asarray(gate, np.float64).T
    if router_bias is not None:
        logits = logits + np.asarray(router_bias, np.float64)[None, :]
    return logits


def score(logits: np.ndarray, score_fn: int) -> np.ndarray:
    """Score function over the logits of each token.

    softmax ([P2] Router table, TopKRouter), sigmoid ([P2] DeepSeek note:
    "fp32 sigmoid"), sqrt(softplus) ([P4] DeepSeek-V4 family; [P3] follow-up
    "sqrtsoftplus scoring")."""
    l = np.asarray(logits, np.float64)
    if score_fn == SCORE_SOFTMAX:
        m = l.max(axis=-1, keepdims=True)
        ex = np.exp(l - m)
        return ex / ex.sum(axis=-1, keepdims=True)
    if score_fn == SCORE_SIGMOID:
        with np.errstate(over="ignore"):
            return 1.0 / (1.0 + np.exp(-l))
    if score_fn == SCORE_SQRTSOFTPLUS:
        # softplus(l) = log(1 + e^l) = max(l, 0) + log1p(e^-|l|)
        return np.sqrt(np.maximum(l, 0.0) + np.log1p(np.exp(-np.abs(l))))
    raise ValueError(f"unknown score function {score_fn}")


# --------------------------------------------------------------------------
# Router, step "select" ([P2] Router table; [P4] select sees the shifted
# scores; [P3] follow-up: the bias is "selection only")
# --------------------------------------------------------------------------

def shift(scores: np.ndarray, expert_bias: Optional[np.ndarray]) -> np.ndarray:
    """choice = scores + expert_bias: the bias steers only the selection
    ([P4]: it changes which experts are picked, not their weights)."""
    if expert_bias is None:
        return np.asarray(scores, np.float64).copy()
    return np.asarray(scores, np.float64) + np.asarray(expert_bias, np.float64)[None, :]


def _k_rounds_argmax(values: np.ndarray, k: int) -> np.ndarray:
    """k rounds of "take the largest remaining entry"; argmax returns the first
    maximum, so ties go to the lower index.  values: [T, N] -> [T, k]."""
    v = np.array(values, np.float64, copy=True)
    rows = np.arange(v.shape[0])
    out = np.empty((v.shape[0], k), np.int64)
    for r in range(k):
        j = np.argmax(v, axis=1)
        out[:, r] = j
        v[rows, j] = -np.inf
    return out


def select_topk(choice: np.ndarray, k: int) -> np.ndarray:
    """Plain top-k over the shifted scores ([P2] Router table, "select")."""
    return _k_rounds_argmax(choice, k)


def group_scores(choice: np.ndarray, n_group: int, group_topn: int) -> np.ndarray:
    """Score of each contiguous expert group: the sum of its ``group_topn``
    largest shifted scores (DeepSeek-V3 group-limited routing, [P2] Router
    table "select" override; [P3] follow-up: the keys use_grouped_topk,
    num_expert_group and topk_group)."""
    t, e = choice.shape
    g = choice.reshape(t, n_group, e // n_group)
    top = -np.sort(-g, axis=2)[:, :, :group_topn]
    return top.sum(axis=2)


def select_group_limited(choice: np.ndarray, k: int, n_group: int,
                         topk_group: int, group_topn: int = 2) -> np.ndarray:
    """Group-limited top-k: keep the ``topk_group`` best groups, make every
    expert outside them unselectable, then plain top-k."""
    t, e = choice.shape
    gsz = e // n_group
    gs = group_scores(choice, n_group, group_topn)
    keep = _k_rounds_argmax(gs, topk_group)
    eligible = np.zeros((t, n_group), bool)
    eligible[np.arange(t)[:, None], keep] = True
    mask = np.repeat(eligible, gsz, axis=1)
    return select_topk(np.where(mask, choice, -np.inf), k)


def select(choice: np.ndarray, recipe: Recipe) -> np.ndarray:
    if recipe.n_group > 1:
        return select_group_limited(choice, recipe.top_k, recipe.n_group,
                                    recipe.topk_group, recipe.group_topn)
    return select_topk(choice, recipe.top_k)


def selection_margin(choice: np.ndarray, idx: np.ndarray, recipe: Recipe) -> np.ndarray:
    """Per token, the smallest gap that decided the selection: between
    consecutive picks, between the last pick and the best eligible non-pick,
    and (group-limited) between the last kept group and the best dropped one.
    A pick that another implementation could flip by rounding the shifted
    scores differently has a margin below that rounding error."""
    t, e = choice.shape
    k = idx.shape[1]
    margins = np.full(t, np.inf)
    if recipe.n_group > 1:
        gs = group_scores(choice, recipe.n_group, recipe.group_topn)
        if recipe.topk_group < recipe.n_group:
            order = -np.sort(-gs, axis=1)
            margins = np.minimum(margins, order[:, recipe.topk_group - 1] - order[:, recipe.topk_group])
        keep = _k_rounds_argmax(gs, recipe.topk_group)
        eligible = np.zeros((t, recipe.n_group), bool)
        eligible[np.arange(t)[:, None], keep] = True
        mask = np.repeat(eligible, e // recipe.n_group, axis=1)
    else:
        mask = np.ones((t, e), bool)
    rows = np.arange(t)[:, None]
    picked = choice[rows, idx]
    if k > 1:
        margins = np.minimum(margins, np.min(picked[:, :-1] - picked[:, 1:], axis=1))
    rest = np.where(mask, choice, -np.inf)
    rest[rows, idx] = -np.inf
    best_rest = rest.max(axis=1)
    margins = np.minimum(margins, picked[:, -1] - best_rest)
    return margins


# --------------------------------------------------------------------------
# Router, step "routing_weights" ([P2] Router table; the 1e-20 note of [P2];
# [P4] DeepSeek-V4 "always renormalized")
# --------------------------------------------------------------------------

def routing_weights(scores: np.ndarray, idx: np.ndarray, recipe: Recipe) -> np.ndarray:
    """Gather the chosen experts' UNSHIFTED scores, renormalise when
    norm_topk_prob (sum + 1e-20), multiply by route_scale."""
    w = np.take_along_axis(np.asarray(scores, np.float64), idx, axis=1)
    if recipe.norm_topk_prob:
        w = w / (w.sum(axis=1, keepdims=True) + recipe.norm_eps)
    return w * recipe.route_scale


def route_from_logits(logits: np.ndarray, recipe: Recipe,
                      expert_bias: Optional[np.ndarray] = None):
    """score -> select(shifted) -> routing_weights, per [P2]'s Router
    template.  Returns (scores, idx [T,K] int64, weights [T,K], choice)."""
    s = score(logits, recipe.score_fn)
    c = shift(s, expert_bias)
    idx = select(c, recipe)
    w = routing_weights(s, idx, recipe)
    return s, idx, w, c


# --------------------------------------------------------------------------
# Token-to-expert grouping ([P2] grouped_mm experts; [P4] tokens_per_expert)
# --------------------------------------------------------------------------

def permute(idx: np.ndarray, num_experts: int):
    """counts[e] = #{(t,k): idx[t,k] = e}; offsets = exclusive prefix sum;
    sorted_pair lists every expert's pairs p = t*K + k in ascending p (a stable
    sort by expert); pair_pos is its inverse permutation."""
    flat = np.asarray(idx, np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=num_experts).astype(np.int64)
    offsets = np.zeros(num_experts + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    sorted_pair = np.argsort(flat, kind="stable").astype(np.int64)
    pair_pos = np.empty_like(sorted_pair)
    pair_pos[sorted_pair] = np.arange(flat.size, dtype=np.int64)
    return counts, offsets, sorted_pair, pair_pos


# --------------------------------------------------------------------------
# Experts ([P1] silu-and-mul / DeepSeek clamped SwiGLU; [P4] fused
# gate_up_proj [2I, H] and down_proj [H, I]); shared expert and combine ([P1],
# [P3])
# --------------------------------------------------------------------------

def silu(v: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def swiglu(g: np.ndarray, u: np.ndarray, limit: float) -> np.ndarray:
    """silu(gate) * up, with DeepSeek's clamp when limit > 0 (gate <= limit,
    |up| <= limit)."""
    if limit > 0:
        g = np.minimum(g, limit)
        u = np.clip(u, -limit, limit)
    return silu(g) * u


def expert_forward(x_rows: np.ndarray, w_gate_up: np.ndarray, w_down: np.ndarray,
                   limit: float) -> np.ndarray:
    """One SwiGLU expert on rows of x: [n, H] -> [n, H].
    w_gate_up [2I, H] (gate rows first), w_down [H, I]."""
    i = w_gate_up.shape[0] // 2
    gu = np.asarray(x_rows, np.float64) @ np.asarray(w_gate_up, np.float64).T
    h = swiglu(gu[:, :i], gu[:, i:], limit)
    return h @ np.asarray(w_down, np.float64).T


def shared_gate(x_rows: np.ndarray, sh_gate: Optional[np.ndarray]) -> np.ndarray:
    """sigmoid(x_t . g) per token when the shared expert is gated, else 1."""
    if sh_gate is None:
        return np.ones(x_rows.shape[0])
    z = np.asarray(x_rows, np.float64) @ np.asarray(sh_gate, np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


ExpertGetter = Callable[[int], Tuple[np.ndarray, np.ndarray]]


def moe_combine_rows(x_rows: np.ndarray, idx_rows: np.ndarray, w_rows: np.ndarray,
                     get_expert: ExpertGetter, limit: float,
                     shared: Optional[Tuple[np.ndarray, np.ndarray]] = None,
                     sh_gate: Optional[np.ndarray] = None) -> np.ndarray:
    """y_t = sum_k w_tk * Expert_{idx_tk}(x_t) + gate_t * Shared(x_t) for the
    given token rows.  The shared expert reads the same x as the routed
    experts ([P1] fix: shared expert computed before the in-place experts
    overwrite their input).  Each expert's weights are fetched once through
    ``get_expert(e) -> (w_gate_up [2I,H], w_down [H,I])``."""
    x_rows = np.asarray(x_rows, np.float64)
    n, k = idx_rows.shape
    outs = np.zeros((n, k, x_rows.shape[1]))
    for e in np.unique(idx_rows):
        wgu, wd = get_expert(int(e))
        rr, kk = np.nonzero(idx_rows == e)
        outs[rr, kk] = expert_forward(x_rows[rr], wgu, wd, limit)
    y = np.zeros((n, x_rows.shape[1]))
    for j in range(k):
        y = y + w_rows[:, j:j + 1] * outs[:, j]
    if shared is not None:
        s = expert_forward(x_rows, shared[0], shared[1], limit)
        y = y + shared_gate(x_rows, sh_gate)[:, None] * s
    return y


def moe_layer(x, gate, w_gate_up, w_down, recipe: Recipe, router_bias=None,
              expert_bias=None, sh_gate_up=None, sh_down=None, sh_gate=None):
    """The whole layer on small inputs: returns dict(logits, scores, choice,
    idx, weights, counts, offsets, sorted_pair, pair_pos, y).  A token count of
    0 routes an empty top-k and returns an empty output ([P1] DraftMoE
    forward: an empty batch gives an empty routing)."""
    x = np.asarray(x, np.float64)
    t, h = x.shape
    e = recipe.num_experts
    logits = router_logits(x, gate, router_bias)
    s, idx, w, c = route_from_logits(logits, recipe, expert_bias) if t else (
        np.zeros((0, e)), np.zeros((0, recipe.top_k), np.int64),
        np.zeros((0, recipe.top_k)), np.zeros((0, e)))
    counts, offsets, sorted_pair, pair_pos = permute(idx, e)
    w_gate_up = np.asarray(w_gate_up, np.float64)
    w_down = np.asarray(w_down, np.float64)
    shared = None if sh_gate_up is None else (np.asarray(sh_gate_up, np.float64),
                                              np.asarray(sh_down, np.float64))
    y = (moe_combine_rows(x, idx, w, lambda j: (w_gate_up[j], w_down[j]),
                          recipe.swiglu_limit, shared, sh_gate)
         if t else np.zeros((0, h)))
    return dict(logits=logits, scores=s, choice=c, idx=idx, weights=w,
                counts=counts, offsets=offsets, sorted_pair=sorted_pair,
                pair_pos=pair_pos, y=y)


# --------------------------------------------------------------------------
# FP4 routed experts ([P4] commit note on the DeepSeek-V4.1 export formats:
# each byte packs the e2m1 codes of two consecutive inputs, the even one in
# its low four bits, and 32 inputs share one e8m0 scale; [P5] MXFP4 commit
# note: uint8 codes [E, N, K//2] and scales [E, N, K//32], output-major).  The layer computes
# with the exactly dequantized weights ([P4]: the import turns them into bf16).
# --------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    """Value of one 4-bit e2m1 code: bit 3 the sign, bits 2..1 a 2-bit
    exponent with bias 1, bit 0 a 1-bit mantissa; exponent 0 is the subnormal
    range (0 or 0.5).  The element format of the OCP microscaling formats."""
    sign = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return sign * 0.5 * m
    return sign * 2.0 ** (e - 1) * (1.0 + 0.5 * m)


def e8m0_value(s: int) -> float:
    """Value of one e8m0 scale byte: 2^(s - 127); 255 encodes NaN."""
    return float("nan") if s == 255 else 2.0 ** (int(s) - 127)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)])
E8M0_TABLE = np.array([e8m0_value(s) for s in range(256)])


def dequant_fp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Exact float64 weights [..., N, K] from codes [..., N, K/2] (uint8, two
    codes per byte along K, the low nibble holding the even index) and scales
    [..., N, K/32] (uint8 e8m0, one per 32 consecutive inputs)."""
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.uint8)
    k = codes.shape[-1] * 2
    assert scales.shape[-1] * 32 == k and scales.shape[:-1] == codes.shape[:-1]
    vals = np.empty(codes.shape[:-1] + (k,))
    vals[..., 0::2] = E2M1_TABLE[codes & 0xF]
    vals[..., 1::2] = E2M1_TABLE[codes >> 4]
    return vals * np.repeat(E8M0_TABLE[scales], 32, axis=-1)


def moe_layer_fp4(x, gate, gu_codes, gu_scales, dn_codes, dn_scales, recipe: Recipe, **kw):
    """The layer with FP4 routed experts: gate_up [E,2I,H/2] codes with
    [E,2I,H/32] scales, down [E,H,I/2] codes with [E,H,I/32] scales; every
    other tensor as in moe_layer()."""
    return moe_layer(x, gate, dequant_fp4(gu_codes, gu_scales), dequant_fp4(dn_codes, dn_scales),
                     recipe, **kw)


# --------------------------------------------------------------------------
# FP8 linears ([P4] commit note on the DeepSeek-V4.1 export formats: the
# official layout keeps its linears as e4m3 with one e8m0 scale per 32 x 32
# block of the weight).  As for FP4, the layer computes with the exactly
# dequantized weights ([P4]: the import turns them into bf16).
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    """Value of one e4m3 byte (the OCP 8-bit floating-point format E4M3, the
    variant without infinities): bit 7 the sign, bits 6..3 a 4-bit exponent
    with bias 7, bits 2..0 the mantissa; exponent 0 is the subnormal range
    (mantissa/8 x 2^-6); exponent 15 with mantissa 7 is NaN, so the largest
    finite value is 1.75 x 2^8 = 448."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)])


def dequant_fp8_blocks(codes: np.ndarray, scales: np.ndarray, block: int = 32) -> np.ndarray:
    """Exact float64 weights [..., N, K] from e4m3 codes [..., N, K] (uint8)
    and e8m0 scales [..., ceil(N/block), ceil(K/block)] (uint8), one scale for
    every block x block tile of the weight."""
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.uint8)
    n, k = codes.shape[-2], codes.shape[-1]
    assert scales.shape[-2] == -(-n // block) and scales.shape[-1] == -(-k // block)
    assert scales.shape[:-2] == codes.shape[:-2]
    s = np.repeat(np.repeat(E8M0_TABLE[scales], block, axis=-2), block, axis=-1)[..., :n, :k]
    return E4M3_TABLE[codes] * s


def moe_layer_fp8(x, gate, gu_codes, gu_scales, dn_codes, dn_scales, recipe: Recipe, **kw):
    """The layer with FP8 routed experts: gate_up [E,2I,H] e4m3 codes with
    [E,2I/32,H/32] scales, down [E,H,I] codes with [E,H/32,I/32] scales;
    every other tensor as in moe_layer()."""
    return moe_layer(x, gate, dequant_fp8_blocks(gu_codes, gu_scales), dequant_fp8_blocks(dn_codes, dn_scales),
                     recipe, **kw)
