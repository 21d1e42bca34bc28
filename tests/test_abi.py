"""The C ABI without a GPU: the library builds, loads, exports every function
include/moe.h declares, and its host-side argument checks refuse bad calls
before touching a device."""
import ctypes

import pytest

from moe_ffn_speculative_gb300 import ops
from moe_ffn_speculative_gb300.build import build


@pytest.fixture(scope="module")
def lib():
    build()
    return ops.lib()


def test_exports_every_declared_function(lib):
    names = ops.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert ops.status_string(ops.MOE_OK) == "MOE_OK"
    assert ops.status_string(ops.MOE_ERR_UNSUPPORTED) == "MOE_ERR_UNSUPPORTED"
    assert ops.status_string(ops.MOE_ERR_DEVICE_TIMEOUT) == "MOE_ERR_DEVICE_TIMEOUT"


def test_route_workspace_size_is_host_only(lib):
    assert lib.moe_route_workspace_bytes(72, 8) >= 256 + 4 * 72 * 8
    assert lib.moe_route_workspace_bytes(-1, 8) == 0


def _forward(lib, rec, T=16, H=64, I=32, x=1 << 20, y=2 << 20, gate=3 << 20, wgu=4 << 20, wd=5 << 20,
             sgu=None, sd=None, Is=0, sg=None):
    return lib.moe_ffn_forward(x, T, H, I, gate, None, None, wgu, wd, sgu, sd, Is, sg, ctypes.byref(rec),
                               6 << 20, 1 << 30, y, None, None, None, None)


def test_recipe_refusals(lib):
    ok = ops.Recipe.make(8, 2)
    bad_k = ops.Recipe.make(8, 9)
    assert _forward(lib, bad_k) == ops.MOE_ERR_UNSUPPORTED
    too_many = ops.Recipe.make(2048, 2)
    assert _forward(lib, too_many) == ops.MOE_ERR_UNSUPPORTED
    groups_not_dividing = ops.Recipe.make(10, 2, n_group=3, topk_group=2)
    assert _forward(lib, groups_not_dividing) == ops.MOE_ERR_UNSUPPORTED
    k_above_groups = ops.Recipe.make(16, 9, n_group=4, topk_group=2)  # only 8 eligible experts
    assert _forward(lib, k_above_groups) == ops.MOE_ERR_UNSUPPORTED
    bad_score = ops.Recipe.make(8, 2, score_fn=7)
    assert _forward(lib, bad_score) == ops.MOE_ERR_INVALID_ARG
    topk_group_too_big = ops.Recipe.make(16, 2, n_group=4, topk_group=5)
    assert _forward(lib, topk_group_too_big) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_ffn_forward(1 << 20, 16, 64, 32, 3 << 20, None, None, 4 << 20, 5 << 20, None, None, 0, None,
                               None, 6 << 20, 1 << 30, 2 << 20, None, None, None, None) == ops.MOE_ERR_INVALID_ARG
    del ok


def test_shape_and_pointer_refusals(lib):
    rec = ops.Recipe.make(8, 2)
    assert _forward(lib, rec, H=60) == ops.MOE_ERR_UNSUPPORTED      # H not a multiple of 8
    assert _forward(lib, rec, I=36) == ops.MOE_ERR_UNSUPPORTED      # I not a multiple of 8
    assert _forward(lib, rec, T=-1) == ops.MOE_ERR_INVALID_ARG
    assert _forward(lib, rec, x=None) == ops.MOE_ERR_INVALID_ARG
    assert _forward(lib, rec, x=(1 << 20) + 2) == ops.MOE_ERR_INVALID_ARG  # misaligned
    assert _forward(lib, rec, y=1 << 20) == ops.MOE_ERR_INVALID_ARG  # y aliases x
    assert _forward(lib, rec, Is=64) == ops.MOE_ERR_INVALID_ARG     # Is without shared weights
    assert _forward(lib, rec, sgu=7 << 20, sd=None, Is=64) == ops.MOE_ERR_INVALID_ARG
    assert _forward(lib, rec, sg=8 << 20) == ops.MOE_ERR_INVALID_ARG  # gate without a shared expert


def test_zero_tokens_launch_nothing(lib):
    rec = ops.Recipe.make(8, 2)
    assert _forward(lib, rec, T=0) == ops.MOE_OK
    assert lib.moe_route_from_logits(None, 0, None, ctypes.byref(rec), None, None, None) == ops.MOE_OK


def test_workspace_refusals_before_any_device_call(lib):
    """A workspace missing, misaligned or smaller than the fixed header is
    refused on the host, before the library asks the device anything."""
    rec = ops.Recipe.make(8, 2)
    args = (1 << 20, 16, 64, 32, 3 << 20, None, None, 4 << 20, 5 << 20, None, None, 0, None, ctypes.byref(rec))
    tail = (2 << 20, None, None, None, None)
    assert lib.moe_ffn_forward(*args, None, 1 << 30, *tail) == ops.MOE_ERR_WORKSPACE
    assert lib.moe_ffn_forward(*args, (6 << 20) + 64, 1 << 30, *tail) == ops.MOE_ERR_WORKSPACE
    assert lib.moe_ffn_forward(*args, 6 << 20, 4096, *tail) == ops.MOE_ERR_WORKSPACE
    # the router: one byte short of moe_route_workspace_bytes
    need = lib.moe_route_workspace_bytes(72, 8)
    assert lib.moe_route(1 << 20, 72, 64, 3 << 20, None, None, ctypes.byref(rec), None, 4 << 20, 5 << 20,
                         6 << 20, need - 1, None) == ops.MOE_ERR_WORKSPACE


def test_route_workspace_size_does_not_depend_on_where_counters_sit(lib):
    """The router's counters sit in a fixed header: the size grows with the
    logits only, by 4 bytes per (token, expert) rounded to 256."""
    base = lib.moe_route_workspace_bytes(0, 8)
    for T, E in [(1, 8), (72, 256), (4096, 64), (65536, 1)]:
        assert lib.moe_route_workspace_bytes(T, E) == base + -(-4 * T * E // 256) * 256


def test_noalloc_router_checks_arguments_first(lib):
    """moe_route_noalloc makes moe_route's checks before it touches its array:
    an invalid recipe is INVALID_ARG (not a size refusal), sizes beyond the
    array are UNSUPPORTED, T = 0 is OK -- none of it needs a device."""
    x, gate, idx, w = 1 << 20, 2 << 20, 3 << 20, 4 << 20
    e0 = ops.Recipe(0, 1, 0, 1, 1, 2, 1, 1e-20, 1.0, 0.0)
    assert lib.moe_route_noalloc(x, 72, 64, gate, None, None, ctypes.byref(e0), None, idx, w, None) == \
        ops.MOE_ERR_INVALID_ARG
    assert lib.moe_route_noalloc(x, 72, 64, gate, None, None, None, None, idx, w, None) == ops.MOE_ERR_INVALID_ARG
    rec = ops.Recipe.make(8, 2)
    assert lib.moe_route_noalloc(None, 72, 64, gate, None, None, ctypes.byref(rec), None, idx, w, None) == \
        ops.MOE_ERR_INVALID_ARG
    assert lib.moe_route_noalloc(x + 2, 72, 64, gate, None, None, ctypes.byref(rec), None, idx, w, None) == \
        ops.MOE_ERR_INVALID_ARG
    assert lib.moe_route_noalloc(x, 4097, 64, gate, None, None, ctypes.byref(rec), None, idx, w, None) == \
        ops.MOE_ERR_UNSUPPORTED
    big = ops.Recipe.make(128, 2)
    assert lib.moe_route_noalloc(x, 4096, 64, gate, None, None, ctypes.byref(big), None, idx, w, None) == \
        ops.MOE_ERR_UNSUPPORTED
    assert lib.moe_route_noalloc(None, 0, 64, None, None, None, ctypes.byref(rec), None, None, None, None) == \
        ops.MOE_OK


def test_block_scaled_refusals_before_any_device_call(lib):
    """moe_ffn_forward_mx / moe_mx_* refuse a bad format, a shape that is not
    a multiple of 128 and a missing workspace on the host."""
    rec = ops.Recipe.make(8, 2)
    assert lib.moe_mx_scales_bytes(ops.FMT_FP4, 8, 4096, 2304, 2304) > 0
    assert lib.moe_mx_scales_bytes(3, 8, 4096, 2304, 0) == 0
    assert lib.moe_mx_scales_bytes(ops.FMT_FP8, 8, 4096 + 64, 2304, 0) == 0

    def fwd(fmt=ops.FMT_FP4, H=256, I=256, Is=0, ws=6 << 20, ws_bytes=1 << 30):
        return lib.moe_ffn_forward_mx(1 << 20, 16, H, I, 2 << 20, None, None, fmt, 3 << 20, 4 << 20, None, None, Is,
                                      None, 5 << 20, 1 << 30, ctypes.byref(rec), ws, ws_bytes, 7 << 20, None, None,
                                      None, None)
    assert fwd(fmt=0) == ops.MOE_ERR_INVALID_ARG
    assert fwd(H=192) == ops.MOE_ERR_UNSUPPORTED
    assert fwd(I=320) == ops.MOE_ERR_UNSUPPORTED
    assert fwd(Is=128) == ops.MOE_ERR_INVALID_ARG  # a shared width without shared weights
    assert fwd(ws=None) == ops.MOE_ERR_WORKSPACE
    assert fwd(ws_bytes=1024) == ops.MOE_ERR_WORKSPACE
    assert lib.moe_mx_prepare_scales(ops.FMT_FP4, 1 << 20, 2 << 20, 8, 4096, 2304, None, None, 0, 3 << 20, 16,
                                     None) == ops.MOE_ERR_WORKSPACE


def test_layer_path_selection():
    """Which entry point a layer's weights take, decided on the host from the
    tensors' presence and shapes (CPU tensors: no library call is made)."""
    from moe_ffn_speculative_gb300 import synthetic as S

    def t(**kw):
        return S.make_inputs(S.LayerConfig("sel", T=2, H=256, E=2, I=256, K=1, seed=3, **kw))

    assert ops.layer_path(t()) == "bf16"
    assert ops.layer_path(t(shared_I=128)) == "bf16"
    # FP4 codes: block-scaled by default, the converter when asked
    assert ops.layer_path(t(expert_format="fp4")) == "mx"
    assert ops.layer_path(t(expert_format="fp4"), mx=False) == "fp4"
    # a bf16 shared expert keeps FP4 on the converter; asking otherwise is refused
    assert ops.layer_path(t(expert_format="fp4", shared_I=128)) == "fp4"
    with pytest.raises(ValueError):
        ops.layer_path(t(expert_format="fp4", shared_I=128), mx=True)
    # an FP8 shared expert or FP8 routed experts: block-scaled only
    assert ops.layer_path(t(expert_format="fp4", shared_I=128, shared_format="fp8")) == "mx"
    assert ops.layer_path(t(expert_format="fp8")) == "mx"
    with pytest.raises(ValueError):
        ops.layer_path(t(expert_format="fp8"), mx=False)
    with pytest.raises(ValueError):
        ops.layer_path(t(expert_format="fp8", shared_I=128))
    # widths the block-scaled path does not take (I = 192) stay on the converter
    d = S.make_inputs(S.LayerConfig("sel", T=2, H=256, E=2, I=192, K=1, expert_format="fp4", seed=3))
    assert ops.layer_path(d) == "fp4"
    # bf16 experts cannot take the block-scaled path
    with pytest.raises(ValueError):
        ops.layer_path(t(), mx=True)


def test_l2_prefetch_refusals(lib):
    """moe_set_l2_prefetch only records ranges (no device access): more than
    eight ranges, missing arrays, a null or misaligned pointer are refused;
    an empty list clears."""
    P = ctypes.c_void_p
    arr = (P * 9)(*([P(0x1000)] * 9))
    sizes = (ctypes.c_size_t * 9)(*([4096] * 9))
    assert lib.moe_set_l2_prefetch(ctypes.cast(arr, P), ctypes.cast(sizes, P), 9) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_set_l2_prefetch(None, None, 1) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_set_l2_prefetch(None, None, -1) == ops.MOE_ERR_INVALID_ARG
    bad = (P * 1)(P(0x1008))
    assert lib.moe_set_l2_prefetch(ctypes.cast(bad, P), ctypes.cast(sizes, P), 1) == ops.MOE_ERR_INVALID_ARG
    null = (P * 1)(P(0))
    assert lib.moe_set_l2_prefetch(ctypes.cast(null, P), ctypes.cast(sizes, P), 1) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_set_l2_prefetch(None, None, 0) == 0


def test_launch_overlap_setting(lib):
    """The per-thread launch-overlap switch takes 0 or 1 and refuses the rest,
    without touching a device."""
    assert lib.moe_set_launch_overlap(2) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_set_launch_overlap(-1) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_set_launch_overlap(0) == ops.MOE_OK
    assert lib.moe_set_launch_overlap(1) == ops.MOE_OK
    ops.set_launch_overlap(False)
    ops.set_launch_overlap(True)
