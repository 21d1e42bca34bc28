"""The device-side failure path, exercised without a fault: the workspace's
start gate (status word 2) is closed from the host, so the expert kernel's
bounded wait at its start runs out (about one second of SM clocks).  The
forward must end on its own with MOE_ERR_DEVICE_TIMEOUT and the gate's info
word -- every CTA raising its abort flag, letting its issued copies land and
freeing its tensor memory -- and, with the gate open again, the next forward
on the same workspace and device must be correct.  Nothing here faults, traps
or waits without a bound."""
import pytest
import torch

from moe_ffn_speculative_gb300 import ops
from moe_ffn_speculative_gb300 import synthetic as S
from moe_ffn_speculative_gb300.build import build

pytestmark = pytest.mark.gpu

CASES = {
    # the fused one-launch kernel (units wait at the gate after the
    # prologue's loads are issued; helpers and combine tasks see the status)
    "slice": (S.LayerConfig("gate_slice", T=72, H=512, E=8, I=384, K=1, seed=51), ops.SCHEDULE_SLICE, None),
    # router launch, then the stream-K expert kernel (every CTA waits)
    "stream_k": (S.LayerConfig("gate_sk", T=64, H=320, E=16, I=160, K=4, shared_I=96, shared_gated=True,
                               seed=52), ops.SCHEDULE_STREAM_K, None),
    # the FP4 expert kernel (converter warps too)
    "fp4": (S.LayerConfig("gate_fp4", T=16, H=128, E=8, I=128, K=2, expert_format="fp4", seed=53),
            ops.SCHEDULE_AUTO, False),
    # the block-scaled kernel (its prologue's image writers and the image
    # gather too), FP4 routed experts and an FP8 shared expert
    "mx": (S.LayerConfig("gate_mx", T=40, H=256, E=8, I=256, K=2, shared_I=128, expert_format="fp4",
                         shared_format="fp8", seed=54), ops.SCHEDULE_AUTO, True),
}


@pytest.fixture(scope="module", autouse=True)
def _library():
    build()
    ops.lib()
    torch.cuda.init()


@pytest.mark.parametrize("name", list(CASES))
def test_closed_start_gate_times_out_and_the_next_forward_is_correct(name):
    cfg, sched, mx = CASES[name]
    d = {k: (None if v is None else v.cuda()) for k, v in S.make_inputs(cfg).items()}
    ops.set_schedule(sched)
    try:
        layer = ops.MoELayer(d, ops.Recipe.from_config(cfg), cfg.T, mx=mx)
        assert layer.mx == bool(mx)
        used = ops.ffn_schedule(cfg.T, cfg.H, cfg.I, cfg.shared_I, layer.recipe, gated=cfg.shared_gated)
        if cfg.expert_format != "fp4":
            assert used == sched
        y_ref = layer.forward(d["x"]).clone()
        torch.cuda.synchronize()
        assert layer.ws.device_status() == (0, 0)

        layer.ws.set_start_gate(True)
        layer.forward(d["x"])
        st, info = layer.ws.device_status()   # synchronises: the forward ended by itself
        assert (st, info) == (ops.MOE_ERR_DEVICE_TIMEOUT, ops.INFO_HOLD)
        assert layer.ws.device_status() == (0, 0)  # read and cleared

        layer.ws.set_start_gate(False)
        for _ in range(2):
            y = layer.forward(d["x"])
            torch.cuda.synchronize()
            assert layer.ws.device_status() == (0, 0)
            assert torch.equal(y, y_ref)
    finally:
        ops.set_schedule(ops.SCHEDULE_AUTO)
