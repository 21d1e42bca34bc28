"""moe_route_noalloc: the router for callers that cannot allocate device memory
when they call it (a serving engine whose memory pool already holds the whole
device, code that must not re-enter its allocator, a C caller without a
device allocator).  Its scratch is a fixed array inside the library, so the
test checks that consecutive calls -- which share that array -- each give the
same routing as moe_route with its own workspace."""
import numpy as np
import pytest
import torch

from moe_ffn_speculative_gb300 import ops
from moe_ffn_speculative_gb300.build import build

pytestmark = pytest.mark.gpu

W_ABS_TOL = 1e-6    # routing weights, as in the parity tests
LOGIT_TOL = 3e-5    # fp32 logits, as in the parity tests


def _case(T, H, E, seed, expert_bias=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16).cuda()
    gate = (torch.randn((E, H), generator=g) * 0.02).to(torch.bfloat16).cuda()
    eb = (torch.randn(E, generator=g) * 0.05).cuda() if expert_bias else None
    return x, gate, eb


def _check_same(rec, x, gate, eb):
    i_ref, w_ref, l_ref = ops.moe_route(x, gate, rec, expert_bias=eb)
    i_na, w_na, l_na = ops.moe_route_noalloc(x, gate, rec, expert_bias=eb)
    torch.cuda.synchronize()
    assert torch.equal(i_na, i_ref)
    assert (w_na - w_ref).abs().max().item() <= W_ABS_TOL
    assert (l_na - l_ref).abs().max().item() <= LOGIT_TOL


def test_noalloc_router_matches_workspace_router_on_consecutive_calls():
    build()
    ops.lib()
    top1 = ops.Recipe.make(8, 1)
    grouped = ops.Recipe.make(256, 8, score_fn=ops.SCORE_SIGMOID, n_group=8, topk_group=4, route_scale=2.5)
    a = _case(72, 4096, 8, seed=1)
    b = _case(100, 7168, 256, seed=3, expert_bias=True)
    _check_same(top1, *a)      # first call
    _check_same(grouped, *b)   # second call reuses the same array
    _check_same(top1, *a)      # and back: nothing left over from the larger call


def _check_same_no_logits(rec, x, gate, eb):
    """With logits_out NULL the fp32 logits live in the library's array."""
    i_ref, w_ref, _ = ops.moe_route(x, gate, rec, expert_bias=eb, want_logits=False)
    i_na, w_na, l_na = ops.moe_route_noalloc(x, gate, rec, expert_bias=eb, want_logits=False)
    torch.cuda.synchronize()
    assert l_na is None
    assert torch.equal(i_na, i_ref)
    assert (w_na - w_ref).abs().max().item() <= W_ABS_TOL


def test_noalloc_router_logits_in_its_own_array():
    """Back-to-back calls whose logits stay inside the array: a decode-sized
    call, one above 1024 tokens (the tiled logits GEMM, then selection on
    8-token blocks), one that fills the array exactly (T*E equal to its
    logits limit), then the small call again, so that leftovers of a larger
    call would show."""
    build()
    ops.lib()
    small = ops.Recipe.make(8, 2)
    mid = ops.Recipe.make(64, 6, score_fn=ops.SCORE_SQRTSOFTPLUS, route_scale=1.5)
    full = ops.Recipe.make(64, 4, score_fn=ops.SCORE_SIGMOID, n_group=8, topk_group=4, route_scale=2.5)
    a = _case(72, 4096, 8, seed=11)
    b = _case(2048, 1024, 64, seed=12, expert_bias=True)
    c = _case(4096, 512, 64, seed=13, expert_bias=True)
    assert 4096 * 64 == 262144  # MOE_NOALLOC_MAX_LOGITS
    _check_same_no_logits(small, *a)
    _check_same_no_logits(mid, *b)
    _check_same_no_logits(full, *c)
    _check_same_no_logits(small, *a)
    _check_same(full, *c)  # and with the logits returned


def test_noalloc_router_refuses_sizes_beyond_its_array():
    build()
    rec = ops.Recipe.make(512, 10)
    x, gate, _ = _case(1024, 64, 512, seed=5)   # T*E = 524288 > MOE_NOALLOC_MAX_LOGITS
    with pytest.raises(ops.MoeError) as e:
        ops.moe_route_noalloc(x, gate, rec)
    assert e.value.status == ops.MOE_ERR_UNSUPPORTED
    x2 = torch.zeros((4097, 64), dtype=torch.bfloat16, device="cuda")  # T > MOE_NOALLOC_MAX_TOKENS
    with pytest.raises(ops.MoeError) as e:
        ops.moe_route_noalloc(x2, gate[:8].contiguous(), ops.Recipe.make(8, 2))
    assert e.value.status == ops.MOE_ERR_UNSUPPORTED
