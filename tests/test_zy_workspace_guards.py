"""Guard bytes around every buffer the library writes: the workspace, y and
the optional routing outputs are views into larger allocations whose margins
hold a known pattern; after each forward (both expert schedules, the
many-token router path, FP4 routed experts) and after moe_route, the margins
must be unchanged.  The library is only ever given pointers inside the
views, so a stray write lands in a margin, never outside this test's memory.
Last, one layer object reused across token counts (its workspace sized for
all of them and zero-filled again when the count changes).
"""
import pytest
import torch

from moe_ffn_speculative_gb300 import ops
from moe_ffn_speculative_gb300 import synthetic as S
from moe_ffn_speculative_gb300.build import build

pytestmark = pytest.mark.gpu

MARGIN = 1 << 16          # bytes on each side of the workspace (keeps its 256-byte alignment)
WS_FILL = 0xA5
Y_FILL = 0x7FA5           # a bf16 NaN bit pattern
I32_FILL = -123456789
F32_FILL = -3.25
ROWS = 4                  # guard rows / elements around the outputs


@pytest.fixture(scope="module", autouse=True)
def _library():
    build()
    ops.lib()
    torch.cuda.init()


class GuardedWorkspace(ops.Workspace):
    """A zero-filled workspace inside an allocation with patterned margins."""

    def __init__(self, nbytes: int, device=None):
        self.nbytes = int(nbytes)
        dev = device or torch.device("cuda", torch.cuda.current_device())
        self.full = torch.zeros(2 * MARGIN + self.nbytes, dtype=torch.uint8, device=dev)
        self.full[:MARGIN] = WS_FILL
        self.full[MARGIN + self.nbytes:] = WS_FILL
        self.buf = self.full[MARGIN:MARGIN + self.nbytes]
        assert self.buf.data_ptr() % 256 == 0

    def margins_intact(self) -> bool:
        return bool((self.full[:MARGIN] == WS_FILL).all().item() and
                    (self.full[MARGIN + self.nbytes:] == WS_FILL).all().item())


def _guarded(shape, dtype, fill):
    """(full, view): `view` has `shape` and starts ROWS rows into `full`."""
    n0 = shape[0]
    full = torch.empty((n0 + 2 * ROWS, *shape[1:]), dtype=dtype, device="cuda")
    if dtype == torch.bfloat16:
        full.view(torch.int16).fill_(fill)
    else:
        full.fill_(fill)
    return full, full[ROWS:ROWS + n0]


def _margins_equal(full, fill):
    a, b = full[:ROWS], full[-ROWS:]
    if full.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    return bool((a == fill).all().item() and (b == fill).all().item())


FP4_TINY = S.LayerConfig("fp4_tiny", T=16, H=128, E=8, I=128, K=2, expert_format="fp4", seed=31)
CASES = {
    "tiny_shared_stream_k": (S.CONFIGS["tiny"].with_(shared_I=32, shared_gated=True, K=2), ops.SCHEDULE_STREAM_K),
    "tiny_shared_slice": (S.CONFIGS["tiny"].with_(shared_I=32, shared_gated=True, K=2), ops.SCHEDULE_SLICE),
    # more than 1024 tokens: the router's logits GEMM, then select and permute
    "many_tokens": (S.LayerConfig("guard_many", T=1100, H=136, E=12, I=64, K=2, shared_I=64, shared_gated=True,
                                  router_bias_std=0.1, seed=41), ops.SCHEDULE_AUTO),
    "fp4_tiny": (FP4_TINY, ops.SCHEDULE_AUTO),
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_writes_stay_inside_their_buffers(name):
    cfg, sched = CASES[name]
    d = {k: (None if v is None else v.cuda()) for k, v in S.make_inputs(cfg).items()}
    rec = ops.Recipe.from_config(cfg)
    fp4 = cfg.expert_format == "fp4"
    ws = GuardedWorkspace(ops.ffn_workspace_bytes(cfg.T, cfg.H, cfg.I, cfg.shared_I, rec))
    y_full, y = _guarded((cfg.T, cfg.H), torch.bfloat16, Y_FILL)
    i_full, idx = _guarded((cfg.T, cfg.K), torch.int32, I32_FILL)
    w_full, w = _guarded((cfg.T, cfg.K), torch.float32, F32_FILL)
    c_full, counts = _guarded((cfg.E,), torch.int32, I32_FILL)
    kw = dict(router_bias=d["router_bias"], expert_bias=d["expert_bias"], sh_gate_up=d["sh_gate_up"],
              sh_down=d["sh_down"], sh_gate=d["sh_gate"], y=y, topk_idx_out=idx, topk_w_out=w, counts_out=counts)
    ops.set_schedule(sched)
    try:
        for _ in range(2):   # the second call runs on the counters the first left behind
            if fp4:
                sc = ops.fp4_prepare_scales(d["w_gate_up_s"], d["w_down_s"])
                ops.moe_ffn_forward_fp4(d["x"], d["gate"], d["w_gate_up_q"], d["w_down_q"], sc, rec, ws, **kw)
            else:
                ops.moe_ffn_forward(d["x"], d["gate"], d["w_gate_up"], d["w_down"], rec, ws, **kw)
            torch.cuda.synchronize()
    finally:
        ops.set_schedule(ops.SCHEDULE_AUTO)
    assert ws.device_status() == (0, 0)
    assert ws.margins_intact(), "a write outside the workspace"
    assert _margins_equal(y_full, Y_FILL), "a write outside y"
    assert _margins_equal(i_full, I32_FILL), "a write outside topk_idx_out"
    assert _margins_equal(w_full, F32_FILL), "a write outside topk_w_out"
    assert _margins_equal(c_full, I32_FILL), "a write outside counts_out"
    assert int(counts.sum().item()) == cfg.T * cfg.K
    assert not torch.isnan(y.float()).any()


def test_route_writes_stay_inside_its_workspace():
    # DeepSeek-V4-style router: 256 experts, top-6, sqrt(softplus), expert bias
    T, H, E = 72, 4096, 256
    g = torch.Generator().manual_seed(42)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16).cuda()
    gate = (torch.randn((E, H), generator=g) * 0.02).to(torch.bfloat16).cuda()
    eb = (torch.randn(E, generator=g) * 0.05).cuda()
    rec = ops.Recipe.make(E, 6, score_fn=ops.SCORE_SQRTSOFTPLUS, route_scale=1.5)
    ws = GuardedWorkspace(ops.lib().moe_route_workspace_bytes(T, E))
    for _ in range(2):
        ops.moe_route(x, gate, rec, expert_bias=eb, ws=ws)
        torch.cuda.synchronize()
    assert ws.device_status() == (0, 0)
    assert ws.margins_intact(), "a write outside the router's workspace"


def _fresh_forward(cfg, d, x):
    layer = ops.MoELayer(d, ops.Recipe.from_config(cfg), max_tokens=x.shape[0])
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.ws.device_status() == (0, 0)
    return y


REUSE = {
    # 12 experts + gated shared expert: the fused kernel at 128 tokens,
    # stream-K with 16-column tiles at 9 and 80-column tiles at 200
    "A": S.LayerConfig("reuse_a", T=200, H=2048, E=12, I=128, K=1, shared_I=128, shared_gated=True,
                       router_bias_std=0.1, seed=43),
    # another shape on the fused kernel (top-1, y written directly)
    "B": S.LayerConfig("reuse_b", T=72, H=512, E=8, I=384, K=1, seed=44),
    # grouped sigmoid top-8 of 64 experts on stream-K, more than 1024 tokens
    # at the largest count (the logits GEMM)
    "C": S.LayerConfig("reuse_c", T=1100, H=320, E=64, I=160, K=8, score_fn=1, n_group=8, topk_group=4,
                       expert_bias_std=0.05, shared_I=96, seed=45),
}
SEQUENCE = [("A", 128), ("B", 72), ("A", 200), ("C", 1100), ("A", 9), ("B", 40), ("C", 17), ("C", 300),
            ("A", 128), ("B", 72)]


def test_one_workspace_serves_every_count_and_shape_without_reset():
    """One workspace, zero-filled once, sized for the largest need, serves a
    sequence of forwards that change the token count, the shape, the recipe
    and the schedule, with no reset in between: every counter sits in the
    fixed header and returns to zero.  Every output equals that of a fresh
    workspace, bit for bit."""
    data = {k: {n: (None if v is None else v.cuda()) for n, v in S.make_inputs(c).items()}
            for k, c in REUSE.items()}
    need = max(ops.ffn_workspace_bytes(T, REUSE[k].H, REUSE[k].I, REUSE[k].shared_I,
                                       ops.Recipe.from_config(REUSE[k])) for k, T in SEQUENCE)
    ws = GuardedWorkspace(need)
    scheds = set()
    for k, T in SEQUENCE:
        cfg, d = REUSE[k], data[k]
        rec = ops.Recipe.from_config(cfg)
        x = d["x"][:T].contiguous()
        scheds.add(ops.ffn_schedule(T, cfg.H, cfg.I, cfg.shared_I, rec, gated=cfg.shared_gated))
        y = ops.moe_ffn_forward(x, d["gate"], d["w_gate_up"], d["w_down"], rec, ws, router_bias=d["router_bias"],
                                expert_bias=d["expert_bias"], sh_gate_up=d["sh_gate_up"], sh_down=d["sh_down"],
                                sh_gate=d["sh_gate"])
        torch.cuda.synchronize()
        assert ws.device_status() == (0, 0), (k, T)
        assert torch.equal(y, _fresh_forward(cfg, d, x)), (k, T)
    assert scheds == {ops.SCHEDULE_SLICE, ops.SCHEDULE_STREAM_K}
    assert ws.margins_intact()


def test_one_router_workspace_serves_every_count_without_reset():
    E, H = 64, 256
    g = torch.Generator().manual_seed(46)
    x = torch.randn((4096, H), generator=g).to(torch.bfloat16).cuda()
    gate = (torch.randn((E, H), generator=g) * 0.02).to(torch.bfloat16).cuda()
    rec = ops.Recipe.make(E, 6, score_fn=ops.SCORE_SQRTSOFTPLUS, route_scale=1.5)
    ws = GuardedWorkspace(ops.lib().moe_route_workspace_bytes(4096, E))
    for T in (9, 4096, 72, 1100, 9):
        xt = x[:T].contiguous()
        i, w, _ = ops.moe_route(xt, gate, rec, ws=ws)
        i_ref, w_ref, _ = ops.moe_route(xt, gate, rec)
        torch.cuda.synchronize()
        assert ws.device_status() == (0, 0), T
        assert torch.equal(i, i_ref) and torch.equal(w, w_ref), T
    assert ws.margins_intact()


def test_layer_reused_across_token_counts():
    """One MoELayer serves token counts that change its schedule and token
    tile: 128 tokens take the fused kernel (12 experts and the gated shared
    expert, untouched experts rare), 9 tokens stream-K with one 16-column
    tile, 200 tokens stream-K with 80-column tiles (a smaller workspace need
    than at 128).  Every forward equals that of a layer built for exactly
    its count."""
    cfg = REUSE["A"]
    d = {k: (None if v is None else v.cuda()) for k, v in S.make_inputs(cfg).items()}
    rec = ops.Recipe.from_config(cfg)
    layer = ops.MoELayer(d, rec, max_tokens=cfg.T)
    for T in (128, 200, 9, 200, 128):
        x = d["x"][:T].contiguous()
        y = layer.forward(x)
        torch.cuda.synchronize()
        assert layer.ws.device_status() == (0, 0)
        assert torch.equal(y, _fresh_forward(cfg, d, x)), f"T={T}"
