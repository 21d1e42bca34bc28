"""GPU checks of the FP4 routed-expert entry points.

The format is DeepSeek-V4.1's official one (SpecForge PR #1073, commit note on
the checkpoint's export formats): e2m1 codes, two per byte along the input
with the even input in the low nibble, one e8m0 scale per 32 inputs.  The
block-scale re-layout is checked element by element; the FP4 expert kernel
itself is not launched (the library refuses every FP4 forward with tokens),
which is checked too.
"""
import numpy as np
import pytest
import torch

from moe_ffn_speculative_gb300 import ops
from moe_ffn_speculative_gb300 import synthetic as S
from moe_ffn_speculative_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    build()
    ops.lib()
    torch.cuda.init()


# ragged gate_up tile (I = 192), ragged down tile (H = 320)
CFG = S.LayerConfig("fp4_ragged", T=37, H=320, E=8, I=192, K=2, shared_I=200, shared_gated=True,
                    expert_format="fp4", seed=32)


def _cuda(d):
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


def test_fp4_scale_layout_round_trip():
    """The re-laid scales hold, for every (expert, tile, k-block), the scale
    pairs of its two 128-row halves; rows past the matrix hold scale 1."""
    d = _cuda(S.make_inputs(CFG))
    sc = ops.fp4_prepare_scales(d["w_gate_up_s"], d["w_down_s"]).cpu().numpy()
    gs, ds = d["w_gate_up_s"].cpu().numpy(), d["w_down_s"].cpu().numpy()
    E, H, I = CFG.E, CFG.H, CFG.I
    mb0, kb0, mb1, kb1 = -(-I // 128), H // 64, -(-H // 256), I // 64
    assert sc.size == E * (mb0 * kb0 + mb1 * kb1) * 512
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


def test_fp4_forward_refuses():
    """Argument errors first; a well-formed FP4 forward with tokens is refused
    (MOE_ERR_UNSUPPORTED) and launches nothing; zero tokens return at once."""
    d = _cuda(S.make_inputs(CFG))
    rec = ops.Recipe.from_config(CFG)
    ws = ops.Workspace(ops.ffn_workspace_bytes(CFG.T, CFG.H, CFG.I, CFG.shared_I, rec))
    sc = ops.fp4_prepare_scales(d["w_gate_up_s"], d["w_down_s"])
    kw = dict(sh_gate_up=d["sh_gate_up"], sh_down=d["sh_down"], sh_gate=d["sh_gate"])
    with pytest.raises(ops.MoeError) as e:
        ops.moe_ffn_forward_fp4(d["x"], d["gate"], d["w_gate_up_q"], d["w_down_q"], sc, rec, ws, **kw)
    assert e.value.status == ops.MOE_ERR_UNSUPPORTED
    # scales buffer too small
    with pytest.raises(ops.MoeError) as e:
        ops.moe_ffn_forward_fp4(d["x"], d["gate"], d["w_gate_up_q"], d["w_down_q"], sc[:256], rec, ws, **kw)
    assert e.value.status == ops.MOE_ERR_INVALID_ARG
    # H not a multiple of 64
    x = torch.zeros((CFG.T, 96), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((CFG.E, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.MoeError) as e:
        ops.moe_ffn_forward_fp4(x, g, d["w_gate_up_q"], d["w_down_q"], sc, rec, ws)
    assert e.value.status == ops.MOE_ERR_UNSUPPORTED
    y = ops.moe_ffn_forward_fp4(d["x"][:0], d["gate"], d["w_gate_up_q"], d["w_down_q"], sc, rec, ws, **kw)
    torch.cuda.synchronize()
    assert y.shape == (0, CFG.H)
    assert ws.device_status() == (0, 0)
