"""Pins of the fp64 oracle against what the pages and the mathematics fix:
hand-worked examples (tests/golden), closed forms, brute force on tiny inputs,
invariants and special cases that reduce to a dense MLP.  Each pin is chosen so
that a plausible mistake in the oracle (a dropped term, a wrong sign, swapped
gate/up halves, a transposed operand, weights from the shifted scores, the
route scale on the shared expert) fails at least one of them."""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- scores

def test_softmax_closed_form():
    s = O.score(np.log([[1.0, 2.0, 3.0, 4.0]]), O.SCORE_SOFTMAX)
    np.testing.assert_allclose(s, [[0.1, 0.2, 0.3, 0.4]], rtol=0, atol=1e-15)
    # shift invariance of softmax
    s2 = O.score(np.log([[1.0, 2.0, 3.0, 4.0]]) + 123.0, O.SCORE_SOFTMAX)
    np.testing.assert_allclose(s2, s, rtol=0, atol=1e-14)


def test_sigmoid_closed_form():
    s = O.score(np.array([[0.0, math.log(3.0), -math.log(3.0), -800.0, 800.0]]), O.SCORE_SIGMOID)
    np.testing.assert_allclose(s, [[0.5, 0.75, 0.25, 0.0, 1.0]], rtol=0, atol=1e-15)


def test_sqrtsoftplus_closed_form():
    l = np.array([[0.0, math.log(3.0), 40.0, -40.0]])
    s = O.score(l, O.SCORE_SQRTSOFTPLUS)
    expect = [math.sqrt(math.log(2.0)), math.sqrt(math.log(4.0)),
              math.sqrt(40.0 + math.log1p(math.exp(-40.0))), math.sqrt(math.log1p(math.exp(-40.0)))]
    np.testing.assert_allclose(s[0], expect, rtol=1e-15, atol=0)
    assert abs(s[0, 3] - math.exp(-20.0)) < 1e-24


# ---------------------------------------------------------------- golden, hand worked

def test_golden_softmax_top2_and_expert_bias():
    g = _golden("router_softmax_top2_hand.json")
    r = O.Recipe(num_experts=4, top_k=g["top_k"], score_fn=g["score_fn"], route_scale=g["route_scale"])
    s, idx, w, _ = O.route_from_logits(np.array(g["logits"]), r)
    np.testing.assert_allclose(s, g["expected_scores"], atol=1e-15)
    assert idx.tolist() == g["expected_idx"]
    np.testing.assert_allclose(w, g["expected_weights"], atol=1e-15)
    s_b, idx_b, w_b, _ = O.route_from_logits(np.array(g["logits"]), r, np.array(g["expert_bias"]))
    assert idx_b.tolist() == g["expected_idx_biased"]
    np.testing.assert_allclose(w_b, g["expected_weights_biased"], atol=1e-15)
    np.testing.assert_array_equal(s_b, s)  # the bias never touches the scores


def test_golden_sigmoid_group_limited():
    g = _golden("router_sigmoid_grouped_hand.json")
    p = np.array([g["p"]])
    logits = np.log(p / (1.0 - p))
    r = O.Recipe(num_experts=8, top_k=g["top_k"], score_fn=g["score_fn"], n_group=g["n_group"],
                 topk_group=g["topk_group"], route_scale=g["route_scale"])
    s, idx, w, c = O.route_from_logits(logits, r)
    np.testing.assert_allclose(O.group_scores(c, 4, 2), g["expected_group_scores"], atol=1e-14)
    assert idx.tolist() == g["expected_idx"]
    np.testing.assert_allclose(w, g["expected_weights"], atol=1e-14)
    plain = O.Recipe(num_experts=8, top_k=2, score_fn=O.SCORE_SIGMOID, route_scale=2.5)
    assert O.route_from_logits(logits, plain)[1].tolist() == g["expected_idx_plain"]


def test_golden_swiglu_clamp():
    g = _golden("swiglu_clamp_hand.json")
    x = np.array(g["x"])
    wgu = np.array(g["w_gate_up"])
    wd = np.array(g["w_down"])
    y_c = O.expert_forward(x, wgu, wd, g["limit"])
    y_u = O.expert_forward(x, wgu, wd, 0.0)
    assert abs(y_c[0, 0] - g["expected_y_clamped"]) < 1e-12
    assert abs(y_u[0, 0] - g["expected_y_unclamped"]) < 1e-12


# ---------------------------------------------------------------- selection: brute force

def _ref_topk(c_row, k):
    return sorted(range(len(c_row)), key=lambda e: (-c_row[e], e))[:k]


def test_topk_equals_full_sort_with_ties():
    rng = np.random.default_rng(7)
    for e in (1, 2, 3, 5, 8, 13, 16):
        for _ in range(40):
            # values from a small set force exact ties
            c = rng.integers(0, 4, size=(6, e)).astype(np.float64) * 0.25
            for k in range(1, e + 1):
                got = O.select_topk(c, k)
                for t in range(c.shape[0]):
                    assert got[t].tolist() == _ref_topk(c[t].tolist(), k)


def _ref_group_limited(c_row, k, n_group, topk_group, topn):
    e = len(c_row)
    gsz = e // n_group
    gscore = [sum(sorted(c_row[g * gsz:(g + 1) * gsz], reverse=True)[:topn]) for g in range(n_group)]
    # brute force over every set of topk_group groups: the kept set is the one
    # whose sorted (-score, index) keys are lexicographically smallest
    best = None
    for combo in itertools.combinations(range(n_group), topk_group):
        key = sorted((-gscore[g], g) for g in combo)
        if best is None or key < best[0]:
            best = (key, combo)
    keep = set(best[1])
    eligible = [j for j in range(e) if j // gsz in keep]
    return sorted(eligible, key=lambda j: (-c_row[j], j))[:k]


def test_group_limited_brute_force():
    rng = np.random.default_rng(11)
    for (e, n_group) in ((8, 4), (8, 2), (12, 3), (16, 4), (16, 8)):
        for topk_group in range(1, n_group + 1):
            gsz = e // n_group
            for k in range(1, topk_group * gsz + 1):
                c = rng.integers(0, 5, size=(5, e)).astype(np.float64) * 0.125
                got = O.select_group_limited(c, k, n_group, topk_group, 2 if gsz >= 2 else 1)
                for t in range(c.shape[0]):
                    ref = _ref_group_limited(c[t].tolist(), k, n_group, topk_group, 2 if gsz >= 2 else 1)
                    assert got[t].tolist() == ref, (e, n_group, topk_group, k, c[t])


def test_group_limited_all_groups_is_plain_topk():
    rng = np.random.default_rng(3)
    for seed in range(20):
        c = rng.normal(size=(9, 32))
        for k in (1, 4, 8):
            np.testing.assert_array_equal(O.select_group_limited(c, k, 8, 8, 2), O.select_topk(c, k))


def test_selection_order_descending():
    rng = np.random.default_rng(5)
    c = rng.normal(size=(50, 64))
    idx = O.select_topk(c, 10)
    picked = np.take_along_axis(c, idx, 1)
    assert np.all(np.diff(picked, axis=1) <= 0)


# ---------------------------------------------------------------- routing weights

@pytest.mark.parametrize("fn", [O.SCORE_SOFTMAX, O.SCORE_SIGMOID, O.SCORE_SQRTSOFTPLUS])
def test_renormalised_weights_sum_to_route_scale(fn):
    rng = np.random.default_rng(fn)
    logits = rng.normal(size=(40, 64)) * 2
    r = O.Recipe(num_experts=64, top_k=6, score_fn=fn, route_scale=1.5)
    _, _, w, _ = O.route_from_logits(logits, r)
    np.testing.assert_allclose(w.sum(axis=1), 1.5, rtol=1e-12)


def test_weights_without_renorm_are_scaled_scores():
    rng = np.random.default_rng(9)
    logits = rng.normal(size=(10, 16))
    r = O.Recipe(num_experts=16, top_k=3, score_fn=O.SCORE_SIGMOID, norm_topk_prob=False, route_scale=2.0)
    s, idx, w, _ = O.route_from_logits(logits, r)
    np.testing.assert_array_equal(w, np.take_along_axis(s, idx, 1) * 2.0)


def test_epsilon_is_bitwise_noop_for_softmax():
    """Sum of the K largest of E softmax probabilities >= K/E >= 1/512, whose
    half-ulp exceeds 1e-20 in fp64 and in fp32."""
    rng = np.random.default_rng(1)
    for e, k in ((8, 1), (8, 2), (512, 10), (256, 8)):
        logits = rng.normal(size=(64, e)) * 3
        a = O.route_from_logits(logits, O.Recipe(e, k, norm_eps=1e-20))[2]
        b = O.route_from_logits(logits, O.Recipe(e, k, norm_eps=0.0))[2]
        np.testing.assert_array_equal(a, b)
        # the same in fp32 arithmetic
        s = O.score(logits, O.SCORE_SOFTMAX).astype(np.float32)
        idx = O.select_topk(s.astype(np.float64), k)
        g = np.take_along_axis(s, idx, 1)
        tot = g.sum(axis=1, keepdims=True, dtype=np.float32)
        np.testing.assert_array_equal(g / (tot + np.float32(1e-20)), g / tot)


def test_epsilon_guards_sigmoid_underflow():
    logits = np.full((1, 4), -800.0)  # every sigmoid underflows to 0
    w = O.route_from_logits(logits, O.Recipe(4, 2, score_fn=O.SCORE_SIGMOID))[2]
    assert np.all(np.isfinite(w)) and np.all(w == 0.0)


def test_top1_renorm_weight_is_route_scale():
    rng = np.random.default_rng(2)
    logits = rng.normal(size=(72, 8)) * 2
    for scale in (1.0, 2.5):
        w = O.route_from_logits(logits, O.Recipe(8, 1, route_scale=scale))[2]
        np.testing.assert_array_equal(w, np.full((72, 1), scale))


def test_route_scale_scales_weights_exactly():
    rng = np.random.default_rng(4)
    logits = rng.normal(size=(30, 32))
    w1 = O.route_from_logits(logits, O.Recipe(32, 4, score_fn=O.SCORE_SIGMOID))[2]
    w25 = O.route_from_logits(logits, O.Recipe(32, 4, score_fn=O.SCORE_SIGMOID, route_scale=2.5))[2]
    np.testing.assert_array_equal(w25, w1 * 2.5)


def test_expert_bias_moves_indices_not_weights():
    rng = np.random.default_rng(6)
    logits = rng.normal(size=(20, 16))
    r = O.Recipe(16, 4, score_fn=O.SCORE_SIGMOID, route_scale=1.0)
    s, idx0, w0, _ = O.route_from_logits(logits, r)
    bias = np.zeros(16)
    bias[15] = 10.0  # promotes expert 15 everywhere
    s1, idx1, w1, _ = O.route_from_logits(logits, r, bias)
    assert np.all(idx1[:, 0] == 15)
    assert not np.array_equal(idx0, idx1)
    gathered = np.take_along_axis(s, idx1, 1)
    np.testing.assert_allclose(w1, gathered / gathered.sum(1, keepdims=True), rtol=1e-15)


def test_router_bias_moves_weights():
    rng = np.random.default_rng(8)
    x = rng.normal(size=(5, 12))
    gate = rng.normal(size=(6, 12)) * 0.1
    rb = rng.normal(size=6)
    l0 = O.router_logits(x, gate)
    l1 = O.router_logits(x, gate, rb)
    for t in range(5):
        for e in range(6):
            ref = sum(x[t, h] * gate[e, h] for h in range(12)) + rb[e]
            assert abs(l1[t, e] - ref) < 1e-12
    w0 = O.route_from_logits(l0, O.Recipe(6, 2))[2]
    w1 = O.route_from_logits(l1, O.Recipe(6, 2))[2]
    assert not np.allclose(w0, w1)


def test_selection_margin_constructed():
    c = np.array([[0.9, 0.5, 0.49, 0.1]])
    idx = O.select_topk(c, 2)
    m = O.selection_margin(c, idx, O.Recipe(4, 2))
    assert abs(m[0] - 0.01) < 1e-12


# ---------------------------------------------------------------- experts and combine

def _dense_swiglu_loops(x, wgu, wd, limit=0.0):
    """Textbook SwiGLU MLP in pure Python loops: gate rows [0, I), up rows
    [I, 2I), down [H, I]."""
    T, H = len(x), len(x[0])
    I = len(wgu) // 2
    out = []
    for t in range(T):
        h = []
        for i in range(I):
            g = sum(wgu[i][j] * x[t][j] for j in range(H))
            u = sum(wgu[I + i][j] * x[t][j] for j in range(H))
            if limit > 0:
                g = min(g, limit)
                u = max(-limit, min(u, limit))
            h.append(g / (1.0 + math.exp(-g)) * u)
        out.append([sum(wd[r][i] * h[i] for i in range(I)) for r in range(H)])
    return out


@pytest.mark.parametrize("limit", [0.0, 0.05])
def test_single_expert_top1_is_dense_mlp(limit):
    rng = np.random.default_rng(12)
    T, H, I = 3, 8, 4
    x = rng.normal(size=(T, H))
    gate = rng.normal(size=(1, H))
    wgu = rng.normal(size=(1, 2 * I, H)) * 0.3
    wd = rng.normal(size=(1, H, I)) * 0.3
    for scale in (1.0, 2.5):
        r = O.Recipe(1, 1, route_scale=scale, swiglu_limit=limit)
        out = O.moe_layer(x, gate, wgu, wd, r)
        np.testing.assert_array_equal(out["weights"], np.full((T, 1), scale))
        ref = np.array(_dense_swiglu_loops(x.tolist(), wgu[0].tolist(), wd[0].tolist(), limit)) * scale
        np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-14)


def test_gate_up_halves_not_interchangeable():
    """Swapping the gate and up halves changes the output (silu is not odd),
    so the dense-MLP pin above fixes the order."""
    rng = np.random.default_rng(13)
    x = rng.normal(size=(2, 6))
    wgu = rng.normal(size=(8, 6))
    wd = rng.normal(size=(6, 4))
    a = O.expert_forward(x, wgu, wd, 0.0)
    b = O.expert_forward(x, np.concatenate([wgu[4:], wgu[:4]]), wd, 0.0)
    assert not np.allclose(a, b)


@pytest.mark.parametrize("gated", [False, True])
def test_shared_expert_gate_and_no_route_scale(gated):
    rng = np.random.default_rng(14)
    T, H, I, Is = 4, 6, 3, 5
    x = rng.normal(size=(T, H))
    gate = rng.normal(size=(1, H))
    wgu = rng.normal(size=(1, 2 * I, H)) * 0.4
    wd = rng.normal(size=(1, H, I)) * 0.4
    sgu = rng.normal(size=(2 * Is, H)) * 0.4
    sd = rng.normal(size=(H, Is)) * 0.4
    sg = rng.normal(size=H) if gated else None
    r = O.Recipe(1, 1, route_scale=2.5)
    y = O.moe_layer(x, gate, wgu, wd, r, sh_gate_up=sgu, sh_down=sd, sh_gate=sg)["y"]
    routed = np.array(_dense_swiglu_loops(x.tolist(), wgu[0].tolist(), wd[0].tolist()))
    shared = np.array(_dense_swiglu_loops(x.tolist(), sgu.tolist(), sd.tolist()))
    if gated:
        gz = np.array([1.0 / (1.0 + math.exp(-sum(x[t, h] * sg[h] for h in range(H)))) for t in range(T)])
    else:
        gz = np.ones(T)
    np.testing.assert_allclose(y, 2.5 * routed + gz[:, None] * shared, rtol=1e-12, atol=1e-13)


def test_topk_combine_against_loops():
    """K = 2 of E = 4: y_t = sum_k w_tk * Expert_{i_tk}(x_t), each expert by loops."""
    rng = np.random.default_rng(15)
    T, H, I, E = 5, 6, 3, 4
    x = rng.normal(size=(T, H))
    gate = rng.normal(size=(E, H))
    wgu = rng.normal(size=(E, 2 * I, H)) * 0.5
    wd = rng.normal(size=(E, H, I)) * 0.5
    out = O.moe_layer(x, gate, wgu, wd, O.Recipe(E, 2))
    for t in range(T):
        ref = np.zeros(H)
        for k in range(2):
            e = out["idx"][t, k]
            ref += out["weights"][t, k] * np.array(
                _dense_swiglu_loops([x[t].tolist()], wgu[e].tolist(), wd[e].tolist())[0])
        np.testing.assert_allclose(out["y"][t], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- permutation

def test_permute_invariants():
    rng = np.random.default_rng(16)
    for (T, K, E) in ((16, 2, 8), (72, 10, 512), (9, 6, 256), (1, 1, 1), (33, 3, 5)):
        idx = np.stack([rng.choice(E, size=K, replace=False) for _ in range(T)])
        counts, offsets, sp, pp = O.permute(idx, E)
        assert counts.sum() == T * K
        np.testing.assert_array_equal(np.sort(sp), np.arange(T * K))
        np.testing.assert_array_equal(pp[sp], np.arange(T * K))
        flat = idx.reshape(-1)
        for e in range(E):
            seg = sp[offsets[e]:offsets[e + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg) > 0)
            assert len(seg) == (flat == e).sum()


def test_empty_input_routes_empty():
    out = O.moe_layer(np.zeros((0, 8)), np.ones((4, 8)), np.ones((4, 6, 8)), np.ones((4, 8, 3)),
                      O.Recipe(4, 2))
    assert out["idx"].shape == (0, 2) and out["y"].shape == (0, 8)
    assert out["counts"].tolist() == [0, 0, 0, 0]


# ---------------------------------------------------------------- FP4 routed experts
# Format of the DeepSeek-V4.1 export (SpecForge PR #1073, commit note on the
# official checkpoint's formats) and the MXFP4 layout of MoE-Infinity PR #143
# (codes [E,N,K//2], scales [E,N,K//32], output-major).

# The sixteen e2m1 values as the OCP microscaling specification lists them
# (codes 0..7 positive, 8..15 their negatives), typed here, not computed.
E2M1_LISTED = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
               -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_code_table():
    assert list(O.E2M1_TABLE) == E2M1_LISTED
    assert math.copysign(1.0, O.E2M1_TABLE[8]) == -1.0  # negative zero


def test_e8m0_matches_library_decoder():
    torch = pytest.importorskip("torch")
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.E8M0_TABLE[:255], lib[:255])
    assert math.isnan(O.E8M0_TABLE[255]) and math.isnan(lib[255])
    assert O.E8M0_TABLE[127] == 1.0 and O.E8M0_TABLE[0] == 2.0 ** -127


def test_fp4_nibble_order_and_scale_blocks():
    # one row of K = 64: byte j holds inputs 2j (low nibble) and 2j+1 (high)
    codes = np.zeros((1, 32), np.uint8)
    codes[0, 0] = 0x21          # input 0 -> code 1 (0.5), input 1 -> code 2 (1.0)
    codes[0, 16] = 0xF7         # input 32 -> code 7 (6.0), input 33 -> code 15 (-6.0)
    scales = np.array([[127, 129]], np.uint8)  # inputs [0,32) x 1, [32,64) x 4
    w = O.dequant_fp4(codes, scales)
    assert w.shape == (1, 64)
    expect = np.zeros(64)
    expect[0], expect[1] = 0.5, 1.0
    expect[32], expect[33] = 24.0, -24.0
    np.testing.assert_array_equal(w[0], expect)


def test_fp4_round_trip_brute_force():
    # an independent encoder: every weight of the form v * 2^k with v in the
    # listed table is encoded by searching the table; dequantizing gives it back
    rng = np.random.default_rng(5)
    n, k = 3, 96
    vals = rng.choice(np.array(E2M1_LISTED[:8] + E2M1_LISTED[9:]), size=(n, k))
    sc = rng.integers(100, 150, size=(n, k // 32)).astype(np.uint8)
    w = vals * np.repeat(2.0 ** (sc.astype(np.int64) - 127), 32, axis=1)
    codes = np.zeros((n, k // 2), np.uint8)
    for r in range(n):
        for j in range(k):
            c = E2M1_LISTED.index(vals[r, j]) if vals[r, j] != 0 else 0
            codes[r, j // 2] |= np.uint8(c << (4 * (j % 2)))
    np.testing.assert_array_equal(O.dequant_fp4(codes, sc), w)


def test_fp4_layer_equals_layer_on_decoded_weights():
    # the FP4 layer is the bf16-formula layer on the decoded weights; the
    # decoding here goes byte by byte through the listed table
    rng = np.random.default_rng(6)
    T, H, E, I, K = 5, 64, 4, 64, 2
    x = rng.standard_normal((T, H))
    gate = rng.standard_normal((E, H)) * 0.1
    gq = rng.integers(0, 256, size=(E, 2 * I, H // 2)).astype(np.uint8)
    gs = rng.integers(118, 122, size=(E, 2 * I, H // 32)).astype(np.uint8)
    dq = rng.integers(0, 256, size=(E, H, I // 2)).astype(np.uint8)
    ds = rng.integers(118, 122, size=(E, H, I // 32)).astype(np.uint8)

    def decode(q, s):
        out = np.zeros(q.shape[:-1] + (q.shape[-1] * 2,))
        for ix in np.ndindex(q.shape):
            b = int(q[ix])
            j = ix[-1]
            sc = 2.0 ** (int(s[ix[:-1] + (2 * j // 32,)]) - 127)
            out[ix[:-1] + (2 * j,)] = E2M1_LISTED[b & 15] * sc
            out[ix[:-1] + (2 * j + 1,)] = E2M1_LISTED[b >> 4] * sc
        return out

    rec = O.Recipe(num_experts=E, top_k=K, score_fn=O.SCORE_SQRTSOFTPLUS, route_scale=1.5, swiglu_limit=10.0)
    a = O.moe_layer_fp4(x, gate, gq, gs, dq, ds, rec)
    b = O.moe_layer(x, gate, decode(gq, gs), decode(dq, ds), rec)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["y"], b["y"])
    # and a swapped nibble order would change the result
    swapped = ((gq & 15) << 4) | (gq >> 4)
    c = O.moe_layer_fp4(x, gate, swapped.astype(np.uint8), gs, dq, ds, rec)
    assert np.abs(c["y"] - a["y"]).max() > 1e-3


# ---------------------------------------------------------------- FP8 linears
# Format of the DeepSeek-V4.1 export (SpecForge PR #1073, commit note on the
# official checkpoint's formats): e4m3 codes, one e8m0 scale per 32 x 32 block.

# e4m3 values the OCP 8-bit floating-point specification fixes, typed here
# from its definition (exponent bias 7, 3 mantissa bits, subnormals below
# 2^-6, S.1111.111 NaN, no infinities), not computed from the oracle's rule.
E4M3_LISTED = {
    0x00: 0.0, 0x01: 0.001953125, 0x02: 0.00390625, 0x07: 0.013671875, 0x08: 0.015625, 0x0F: 0.029296875,
    0x30: 0.5, 0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x48: 4.0, 0x50: 8.0, 0x70: 128.0,
    0x77: 240.0, 0x78: 256.0, 0x7D: 416.0, 0x7E: 448.0,
    0x80: -0.0, 0x81: -0.001953125, 0xB8: -1.0, 0xC0: -2.0, 0xFE: -448.0,
}


def test_e4m3_listed_values():
    for code, v in E4M3_LISTED.items():
        assert O.E4M3_TABLE[code] == v, hex(code)
    assert math.copysign(1.0, O.E4M3_TABLE[0x80]) == -1.0
    assert math.isnan(O.E4M3_TABLE[0x7F]) and math.isnan(O.E4M3_TABLE[0xFF])
    assert np.nanmax(O.E4M3_TABLE) == 448.0 and np.nanmin(O.E4M3_TABLE) == -448.0


def test_e4m3_matches_library_decoder():
    torch = pytest.importorskip("torch")
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(lib)
    np.testing.assert_array_equal(O.E4M3_TABLE[finite], lib[finite])
    np.testing.assert_array_equal(np.isnan(O.E4M3_TABLE), np.isnan(lib))


def test_fp8_32x32_block_scales():
    # a 64 x 96 weight of ones (code 0x38): each 32 x 32 block takes its own
    # scale; the last column block is whole, rows and columns map as written
    codes = np.full((64, 96), 0x38, np.uint8)
    scales = np.array([[126, 127, 128], [129, 130, 131]], np.uint8)
    w = O.dequant_fp8_blocks(codes, scales)
    for bi in range(2):
        for bj in range(3):
            blk = w[32 * bi:32 * bi + 32, 32 * bj:32 * bj + 32]
            assert (blk == 2.0 ** (int(scales[bi, bj]) - 127)).all()
    # a ragged shape: 40 x 40 uses ceil(40/32) = 2 scales per dimension
    w2 = O.dequant_fp8_blocks(np.full((40, 40), 0x40, np.uint8), np.array([[127, 128], [129, 130]], np.uint8))
    assert w2[0, 0] == 2.0 and w2[0, 39] == 4.0 and w2[39, 0] == 8.0 and w2[39, 39] == 16.0


def test_fp8_layer_equals_layer_on_decoded_weights():
    # the FP8 layer is the bf16-formula layer on the decoded weights; here
    # decoded element by element through the listed rule and the block index
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    T, H, E, I, K = 5, 64, 4, 64, 2
    x = rng.standard_normal((T, H))
    gate = rng.standard_normal((E, H)) * 0.1
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    gq = rng.choice(finite, size=(E, 2 * I, H))
    gs = rng.integers(112, 118, size=(E, 2 * I // 32, H // 32)).astype(np.uint8)
    dq = rng.choice(finite, size=(E, H, I))
    ds = rng.integers(112, 118, size=(E, H // 32, I // 32)).astype(np.uint8)

    def decode(q, s):
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        out = np.empty(q.shape)
        for ix in np.ndindex(q.shape):
            out[ix] = v[ix] * 2.0 ** (int(s[ix[:-2] + (ix[-2] // 32, ix[-1] // 32)]) - 127)
        return out

    rec = O.Recipe(num_experts=E, top_k=K, score_fn=O.SCORE_SQRTSOFTPLUS, route_scale=1.5, swiglu_limit=10.0)
    a = O.moe_layer_fp8(x, gate, gq, gs, dq, ds, rec)
    b = O.moe_layer(x, gate, decode(gq, gs), decode(dq, ds), rec)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["y"], b["y"])
    # the row blocks' scales taken in the wrong order would change the result
    c = O.moe_layer(x, gate, O.dequant_fp8_blocks(gq, gs[..., ::-1, :]), O.dequant_fp8_blocks(dq, ds), rec)
    assert np.abs(c["y"] - a["y"]).max() > 1e-3


# ---------------------------------------------------------------------------
# selection margin: perturbations below it keep the selection, and for plain
# top-k one of its size flips it (brute force on small random scores)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n_group,topk_group", [(1, 1), (4, 2), (8, 3)])
def test_selection_margin_bounds_the_perturbations_that_keep_the_selection(n_group, topk_group):
    rng = np.random.default_rng(31 + n_group)
    E, K, T = 16 if n_group < 8 else 32, 4, 40
    rec = O.Recipe(num_experts=E, top_k=K, n_group=n_group, topk_group=topk_group)
    choice = rng.standard_normal((T, E))
    idx = O.select(choice, rec)
    m = O.selection_margin(choice, idx, rec)
    assert (m > 0).all()
    # every shifted score moved by at most m/4.01: a group score (a sum of
    # two scores) by at most m/2.005, so no gap of size >= m can close
    for _ in range(200):
        d = rng.uniform(-1.0, 1.0, (T, E)) * (m[:, None] / 4.01)
        np.testing.assert_array_equal(O.select(choice + d, rec), idx)
    if n_group == 1:
        # the two scores across the smallest gap, moved by 0.51 m towards each
        # other, swap (two picks change order, or a pick leaves the set)
        rows = np.arange(T)
        picked = choice[rows[:, None], idx]
        rest = choice.copy()
        rest[rows[:, None], idx] = -np.inf
        flipped = 0
        for t in range(T):
            gaps = list(picked[t, :-1] - picked[t, 1:]) + [picked[t, -1] - rest[t].max()]
            j = int(np.argmin(gaps))
            assert gaps[j] == pytest.approx(m[t])
            hi = idx[t, j]
            lo = idx[t, j + 1] if j < K - 1 else int(np.argmax(rest[t]))
            c = choice[t].copy()
            c[hi] -= 0.51 * m[t]
            c[lo] += 0.51 * m[t]
            flipped += not np.array_equal(O.select(c[None, :], rec)[0], idx[t])
        assert flipped == T
