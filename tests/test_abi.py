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
