"""Python binding of libmoe_gb300.so (ctypes).

Argument marshalling only: torch supplies device memory and the stream, every
step of the layer runs in the library's CUDA kernels.  There is no fallback:
when the library is missing or the device is not a CUDA GPU the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

(MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE_TIMEOUT,
 MOE_ERR_DEVICE_RANGE) = range(7)
SCORE_SOFTMAX, SCORE_SIGMOID, SCORE_SQRTSOFTPLUS = 0, 1, 2
# the workspace's start gate (include/moe.h) and the info word of its timeout
WS_HOLD_OFFSET = 8
INFO_HOLD = 15
# routed-expert formats of the block-scaled path
FMT_FP4, FMT_FP8 = 1, 2


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class Recipe(ctypes.Structure):
    """Mirror of ``moe_recipe`` in include/moe.h."""

    _fields_ = [
        ("num_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("score_fn", ctypes.c_int32),
        ("n_group", ctypes.c_int32),
        ("topk_group", ctypes.c_int32),
        ("group_topn", ctypes.c_int32),
        ("norm_topk_prob", ctypes.c_int32),
        ("norm_eps", ctypes.c_float),
        ("route_scale", ctypes.c_float),
        ("swiglu_limit", ctypes.c_float),
    ]

    @classmethod
    def make(cls, num_experts, top_k, score_fn=SCORE_SOFTMAX, n_group=1, topk_group=1, group_topn=2,
             norm_topk_prob=True, norm_eps=1e-20, route_scale=1.0, swiglu_limit=0.0) -> "Recipe":
        return cls(num_experts, top_k, score_fn, n_group, topk_group if n_group > 1 else 1, group_topn,
                   1 if norm_topk_prob else 0, norm_eps, route_scale, swiglu_limit)

    @classmethod
    def from_config(cls, cfg) -> "Recipe":
        """From a ``synthetic.LayerConfig``."""
        return cls.make(cfg.E, cfg.K, cfg.score_fn, cfg.n_group, cfg.topk_group, cfg.group_topn,
                        cfg.norm_topk_prob, cfg.norm_eps, cfg.route_scale, cfg.swiglu_limit)


_lib_handle: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_route_workspace_bytes": (_SZ, [_I, _I]),
    "moe_route": (_I, [_P, _I, _I, _P, _P, _P, ctypes.POINTER(Recipe), _P, _P, _P, _P, _SZ, _P]),
    "moe_route_noalloc": (_I, [_P, _I, _I, _P, _P, _P, ctypes.POINTER(Recipe), _P, _P, _P, _P]),
    "moe_route_from_logits": (_I, [_P, _I, _P, ctypes.POINTER(Recipe), _P, _P, _P]),
    "moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_ffn_workspace_bytes": (_SZ, [_I, _I, _I, _I, ctypes.POINTER(Recipe)]),
    "moe_workspace_init": (_I, [_P, _SZ, _P]),
    "moe_ffn_forward": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, ctypes.POINTER(Recipe),
                             _P, _SZ, _P, _P, _P, _P, _P]),
    "moe_get_device_status": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "moe_set_profile_events": (None, [_P, _I]),
    "moe_set_l2_prefetch": (_I, [_P, _P, _I]),
    "moe_set_schedule": (_I, [_I]),
    "moe_set_launch_overlap": (_I, [_I]),
    "moe_ffn_schedule": (_I, [_I, _I, _I, _I, ctypes.POINTER(Recipe), _I]),
    "moe_fp4_scales_bytes": (_SZ, [_I, _I, _I]),
    "moe_fp4_prepare_scales": (_I, [_P, _P, _I, _I, _I, _P, _SZ, _P]),
    "moe_ffn_forward_fp4": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _I, _P,
                                 ctypes.POINTER(Recipe), _P, _SZ, _P, _P, _P, _P, _P]),
    "moe_mx_scales_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_mx_prepare_scales": (_I, [_I, _P, _P, _I, _I, _I, _P, _P, _I, _P, _SZ, _P]),
    "moe_ffn_forward_mx": (_I, [_P, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _P, _SZ,
                                ctypes.POINTER(Recipe), _P, _SZ, _P, _P, _P, _P, _P]),
}

SCHEDULE_AUTO, SCHEDULE_STREAM_K, SCHEDULE_SLICE = 0, 1, 2
SCHEDULE_NAMES = {SCHEDULE_STREAM_K: "stream_k", SCHEDULE_SLICE: "slice"}


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with moe_ffn_speculative_gb300.build.build()")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = h
    return _lib_handle


def header_functions():
    """Names of the functions include/moe.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensor is not on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("tensor is not contiguous")


def _u16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return t


# --------------------------------------------------------------------------- workspaces

class Workspace:
    """A zero-filled device workspace owned by torch's allocator."""

    def __init__(self, nbytes: int, device=None):
        self.nbytes = int(nbytes)
        self.buf = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8,
                               device=device or torch.device("cuda", torch.cuda.current_device()))

    def ptr(self) -> int:
        return self.buf.data_ptr()

    def reset(self, stream=None) -> None:
        """Zero-fill again (moe_workspace_init), as after a device-side error."""
        _check(lib().moe_workspace_init(self.ptr(), self.nbytes, _stream(stream)), "moe_workspace_init")

    def set_start_gate(self, closed: bool, stream=None) -> None:
        """Close (non-zero) or open (zero) the workspace's start gate."""
        v = torch.tensor([1 if closed else 0], dtype=torch.int32, device=self.buf.device)
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            self.buf[WS_HOLD_OFFSET:WS_HOLD_OFFSET + 4].copy_(v.view(torch.uint8))

    def device_status(self, stream=None) -> Tuple[int, int]:
        info = ctypes.c_int32(0)
        st = lib().moe_get_device_status(self.ptr(), _stream(stream), ctypes.byref(info))
        return st, info.value


def ffn_workspace_bytes(T: int, H: int, I: int, Is: int, recipe: Recipe) -> int:
    n = lib().moe_ffn_workspace_bytes(T, H, I, Is, ctypes.byref(recipe))
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_ffn_workspace_bytes")
    return n


def ffn_workspace_bytes_upto(max_tokens: int, H: int, I: int, Is: int, recipe: Recipe) -> int:
    """Bytes of a workspace that serves every token count 1..max_tokens: the
    size for exactly T is not monotone in T (above 128 tokens the token tile
    narrows to about four times an expert's mean load, shrinking its
    partial-accumulator region)."""
    n = 0
    for T in range(1, max_tokens + 1):
        n = max(n, ffn_workspace_bytes(T, H, I, Is, recipe))
    return n


# --------------------------------------------------------------------------- entry points

def moe_route(x, gate, recipe: Recipe, router_bias=None, expert_bias=None, ws: Workspace = None,
              want_logits=True, stream=None):
    """-> (topk_idx int32 [T,K], topk_w fp32 [T,K], logits fp32 [T,E] or None)."""
    _need_cuda(x, gate, router_bias, expert_bias)
    T, H = x.shape
    E, K = recipe.num_experts, recipe.top_k
    dev = x.device
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if want_logits else None
    if ws is None:
        ws = Workspace(lib().moe_route_workspace_bytes(T, E), dev)
    _check(lib().moe_route(_ptr(_u16(x)), T, H, _ptr(_u16(gate)), _ptr(router_bias), _ptr(expert_bias),
                           ctypes.byref(recipe), _ptr(logits), _ptr(idx), _ptr(w), ws.ptr(), ws.nbytes,
                           _stream(stream)), "moe_route")
    return idx, w, logits


def moe_route_noalloc(x, gate, recipe: Recipe, router_bias=None, expert_bias=None, want_logits=True,
                      stream=None):
    """moe_route with the library's fixed scratch array instead of a workspace.
    -> (topk_idx int32 [T,K], topk_w fp32 [T,K], logits fp32 [T,E] or None)."""
    _need_cuda(x, gate, router_bias, expert_bias)
    T, H = x.shape
    E, K = recipe.num_experts, recipe.top_k
    dev = x.device
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if want_logits else None
    _check(lib().moe_route_noalloc(_ptr(_u16(x)), T, H, _ptr(_u16(gate)), _ptr(router_bias), _ptr(expert_bias),
                                   ctypes.byref(recipe), _ptr(logits), _ptr(idx), _ptr(w), _stream(stream)),
           "moe_route_noalloc")
    return idx, w, logits


def moe_route_from_logits(logits, recipe: Recipe, expert_bias=None, stream=None):
    """-> (topk_idx int32 [T,K], topk_w fp32 [T,K])."""
    _need_cuda(logits, expert_bias)
    T = logits.shape[0]
    K = recipe.top_k
    idx = torch.empty((T, K), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, K), dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_from_logits(_ptr(logits), T, _ptr(expert_bias), ctypes.byref(recipe), _ptr(idx),
                                       _ptr(w), _stream(stream)), "moe_route_from_logits")
    return idx, w


def moe_permute(topk_idx, num_experts: int, stream=None):
    """-> (counts [E], offsets [E+1], sorted_pair [T*K], pair_pos [T*K]), int32."""
    _need_cuda(topk_idx)
    T, K = topk_idx.shape
    dev = topk_idx.device
    counts = torch.empty(num_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(T * K, dtype=torch.int32, device=dev)
    pp = torch.empty(T * K, dtype=torch.int32, device=dev)
    _check(lib().moe_permute(_ptr(topk_idx), T, K, num_experts, _ptr(counts), _ptr(offsets), _ptr(sp), _ptr(pp),
                             None, 0, _stream(stream)), "moe_permute")
    return counts, offsets, sp, pp


def moe_ffn_forward(x, gate, w_gate_up, w_down, recipe: Recipe, ws: Workspace, router_bias=None,
                    expert_bias=None, sh_gate_up=None, sh_down=None, sh_gate=None, y=None,
                    topk_idx_out=None, topk_w_out=None, counts_out=None, stream=None):
    """The whole layer; returns y [T,H] bf16."""
    _need_cuda(x, gate, w_gate_up, w_down, router_bias, expert_bias, sh_gate_up, sh_down, sh_gate, y,
               topk_idx_out, topk_w_out, counts_out)
    T, H = x.shape
    I = w_down.shape[2]
    Is = 0 if sh_gate_up is None else sh_down.shape[1]
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_ffn_forward(
        _ptr(_u16(x)), T, H, I, _ptr(_u16(gate)), _ptr(router_bias), _ptr(expert_bias), _ptr(_u16(w_gate_up)),
        _ptr(_u16(w_down)), _ptr(sh_gate_up), _ptr(sh_down), Is, _ptr(sh_gate), ctypes.byref(recipe), ws.ptr(),
        ws.nbytes, _ptr(y), _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(counts_out), _stream(stream)),
        "moe_ffn_forward")
    return y


def _u8(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.uint8:
        raise TypeError("expected a uint8 tensor")
    return t


def fp4_prepare_scales(w_gate_up_s, w_down_s, stream=None) -> torch.Tensor:
    """The e8m0 scales [E,2I,H/32] and [E,H,I/32] re-laid for
    moe_ffn_forward_fp4 (once per set of weights); returns the uint8 buffer."""
    _need_cuda(w_gate_up_s, w_down_s)
    E, H = w_down_s.shape[0], w_down_s.shape[1]
    I = w_gate_up_s.shape[1] // 2
    n = lib().moe_fp4_scales_bytes(E, H, I)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED, "moe_fp4_scales_bytes")
    out = torch.empty(n, dtype=torch.uint8, device=w_down_s.device)
    _check(lib().moe_fp4_prepare_scales(_ptr(_u8(w_gate_up_s)), _ptr(_u8(w_down_s)), E, H, I, _ptr(out), n,
                                        _stream(stream)), "moe_fp4_prepare_scales")
    return out


def moe_ffn_forward_fp4(x, gate, w_gate_up_q, w_down_q, scales, recipe: Recipe, ws: Workspace, router_bias=None,
                        expert_bias=None, sh_gate_up=None, sh_down=None, sh_gate=None, y=None,
                        topk_idx_out=None, topk_w_out=None, counts_out=None, stream=None):
    """The whole layer with FP4 routed experts (codes [E,2I,H/2], [E,H,I/2];
    ``scales`` from fp4_prepare_scales); returns y [T,H] bf16."""
    _need_cuda(x, gate, w_gate_up_q, w_down_q, scales, router_bias, expert_bias, sh_gate_up, sh_down, sh_gate, y,
               topk_idx_out, topk_w_out, counts_out)
    T, H = x.shape
    I = w_down_q.shape[2] * 2
    Is = 0 if sh_gate_up is None else sh_down.shape[1]
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_ffn_forward_fp4(
        _ptr(_u16(x)), T, H, I, _ptr(_u16(gate)), _ptr(router_bias), _ptr(expert_bias), _ptr(_u8(w_gate_up_q)),
        _ptr(_u8(w_down_q)), _ptr(_u8(scales)), scales.numel(), _ptr(sh_gate_up), _ptr(sh_down), Is, _ptr(sh_gate),
        ctypes.byref(recipe), ws.ptr(), ws.nbytes, _ptr(y), _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(counts_out),
        _stream(stream)), "moe_ffn_forward_fp4")
    return y


def mx_format(t: dict) -> int:
    """Routed-expert format of a block-scaled layer's tensors: FP4 scales
    [E,2I,H/32] have a row per weight row, FP8 scales [E,2I/32,H/32] one per
    32 rows."""
    return FMT_FP4 if t["w_gate_up_s"].shape[1] == t["w_gate_up_q"].shape[1] else FMT_FP8


def mx_dims(t: dict):
    """(E, H, I, Is) of a block-scaled layer's tensors."""
    q = t["w_gate_up_q"]
    E, I = q.shape[0], q.shape[1] // 2
    H = q.shape[2] * (2 if mx_format(t) == FMT_FP4 else 1)
    Is = 0 if t.get("sh_gate_up_q") is None else t["sh_gate_up_q"].shape[0] // 2
    return E, H, I, Is


def mx_prepare_scales(t: dict, stream=None) -> torch.Tensor:
    """The weight scales of a block-scaled layer (routed w_gate_up_s, w_down_s,
    shared sh_gate_up_s, sh_down_s) re-laid for moe_ffn_forward_mx (once per
    set of weights); returns the uint8 buffer."""
    fmt = mx_format(t)
    E, H, I, Is = mx_dims(t)
    _need_cuda(t["w_gate_up_s"], t["w_down_s"], t.get("sh_gate_up_s"), t.get("sh_down_s"))
    n = lib().moe_mx_scales_bytes(fmt, E, H, I, Is)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED, "moe_mx_scales_bytes")
    out = torch.empty(n, dtype=torch.uint8, device=t["w_down_s"].device)
    _check(lib().moe_mx_prepare_scales(fmt, _ptr(_u8(t["w_gate_up_s"])), _ptr(_u8(t["w_down_s"])), E, H, I,
                                       _ptr(t.get("sh_gate_up_s")), _ptr(t.get("sh_down_s")), Is, _ptr(out), n,
                                       _stream(stream)), "moe_mx_prepare_scales")
    return out


def moe_ffn_forward_mx(x, gate, routed_fmt: int, w_gate_up_q, w_down_q, scales, recipe: Recipe, ws: Workspace,
                       I: int, router_bias=None, expert_bias=None, sh_gate_up_q=None, sh_down_q=None, sh_gate=None,
                       y=None, topk_idx_out=None, topk_w_out=None, counts_out=None, stream=None):
    """The whole layer with block-scaled experts (FP4 or FP8 routed, FP8
    shared); returns y [T,H] bf16."""
    _need_cuda(x, gate, w_gate_up_q, w_down_q, scales, router_bias, expert_bias, sh_gate_up_q, sh_down_q, sh_gate, y,
               topk_idx_out, topk_w_out, counts_out)
    T, H = x.shape
    Is = 0 if sh_gate_up_q is None else sh_gate_up_q.shape[0] // 2
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_ffn_forward_mx(
        _ptr(_u16(x)), T, H, I, _ptr(_u16(gate)), _ptr(router_bias), _ptr(expert_bias), int(routed_fmt),
        _ptr(_u8(w_gate_up_q)), _ptr(_u8(w_down_q)), _ptr(sh_gate_up_q), _ptr(sh_down_q), Is, _ptr(sh_gate),
        _ptr(_u8(scales)), scales.numel(), ctypes.byref(recipe), ws.ptr(), ws.nbytes, _ptr(y), _ptr(topk_idx_out),
        _ptr(topk_w_out), _ptr(counts_out), _stream(stream)), "moe_ffn_forward_mx")
    return y


def set_schedule(schedule: int) -> None:
    """Expert schedule of later moe_ffn_forward calls on this thread:
    SCHEDULE_AUTO, SCHEDULE_STREAM_K or SCHEDULE_SLICE."""
    _check(lib().moe_set_schedule(int(schedule)), "moe_set_schedule")


def set_launch_overlap(enable: bool) -> None:
    """Whether later fused-schedule launches on this thread overlap the
    previous kernel on their stream (True, the default) or are cooperative
    launches (False); both compute the same bits."""
    _check(lib().moe_set_launch_overlap(1 if enable else 0), "moe_set_launch_overlap")


def ffn_schedule(T: int, H: int, I: int, Is: int, recipe: Recipe, gated: bool = False) -> int:
    """The schedule moe_ffn_forward would run for this shape (SCHEDULE_STREAM_K
    or SCHEDULE_SLICE)."""
    s = lib().moe_ffn_schedule(T, H, I, Is, ctypes.byref(recipe), 1 if gated else 0)
    if s < 0:
        raise MoeError(1, "moe_ffn_schedule")
    return s


def set_l2_prefetch(tensors) -> None:
    """The next forward on this thread prefetches these tensors' bytes into
    L2 in its expert kernel's tail (moe_set_l2_prefetch); None or [] clears."""
    ts = [t for t in (tensors or []) if t is not None]
    _need_cuda(*ts)
    ptrs = (ctypes.c_void_p * max(1, len(ts)))(*[t.data_ptr() for t in ts])
    sizes = (ctypes.c_size_t * max(1, len(ts)))(*[t.numel() * t.element_size() for t in ts])
    _check(lib().moe_set_l2_prefetch(ctypes.cast(ptrs, ctypes.c_void_p), ctypes.cast(sizes, ctypes.c_void_p),
                                     len(ts)), "moe_set_l2_prefetch")


def set_profile_events(events) -> None:
    """events: a list of torch.cuda.Event (pairs around each launch) or None."""
    global _profile_keepalive
    if not events:
        lib().moe_set_profile_events(None, 0)
        _profile_keepalive = None
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _profile_keepalive = arr
    lib().moe_set_profile_events(ctypes.cast(arr, ctypes.c_void_p), len(events) // 2)


_profile_keepalive = None


def layer_path(tensors: dict, mx: Optional[bool] = None) -> str:
    """Which entry point runs a layer with these weights: "bf16"
    (moe_ffn_forward), "mx" (moe_ffn_forward_mx: FP4 or FP8 routed codes,
    no shared expert or an FP8 one) or "fp4" (moe_ffn_forward_fp4: FP4
    routed codes, no shared expert or a bf16 one).  mx=None picks the
    block-scaled path wherever it takes the layer (H, I and the shared
    expert's width multiples of 128, no bf16 shared expert); True / False
    ask for it or for the converter path.  Raises ValueError for weights
    that no path takes as asked."""
    if tensors.get("w_down_q") is None:
        if mx:
            raise ValueError("the block-scaled path takes coded routed experts (w_gate_up_q, w_down_q)")
        return "bf16"
    bf16_shared = tensors.get("sh_gate_up") is not None
    fp8_shared = tensors.get("sh_gate_up_q") is not None
    if bf16_shared and fp8_shared:
        raise ValueError("both a bf16 and an FP8 shared expert given")
    fmt = mx_format(tensors)
    if mx is None:
        _, H, I, Is = mx_dims(tensors)
        fits = H % 128 == 0 and I % 128 == 0 and Is % 128 == 0
        mx = fmt == FMT_FP8 or fp8_shared or (fits and not bf16_shared)
    if mx and bf16_shared:
        raise ValueError("the block-scaled path takes an FP8 shared expert (sh_gate_up_q), not a bf16 one")
    if not mx and (fmt == FMT_FP8 or fp8_shared):
        raise ValueError("FP8 weights run only on the block-scaled path")
    return "mx" if mx else "fp4"


class MoELayer:
    """Weights of one layer plus its workspace; ``forward(x)`` runs the layer."""

    def __init__(self, tensors: dict, recipe: Recipe, max_tokens: int, mx: Optional[bool] = None):
        """Routed experts as bf16 (w_gate_up, w_down), or as codes
        (w_gate_up_q, w_down_q with scales w_gate_up_s, w_down_s, re-laid once
        here).  The entry point is chosen by layer_path(tensors, mx): coded
        weights take the block-scaled path (moe_ffn_forward_mx) wherever it
        takes the layer, else FP4 codes take moe_ffn_forward_fp4."""
        self.t = tensors
        self.recipe = recipe
        path = layer_path(tensors, mx)
        self.mx = path == "mx"
        self.fp4 = path == "fp4"
        if self.mx:
            self.fmt = mx_format(tensors)
            _, self.H, self.I, self.Is = mx_dims(tensors)
            self.scales = mx_prepare_scales(tensors)
        elif self.fp4:
            self.H = tensors["w_down_q"].shape[1]
            self.I = tensors["w_down_q"].shape[2] * 2
            self.scales = fp4_prepare_scales(tensors["w_gate_up_s"], tensors["w_down_s"])
        else:
            self.H = tensors["w_down"].shape[1]
            self.I = tensors["w_down"].shape[2]
        if not self.mx:
            self.Is = 0 if tensors.get("sh_gate_up") is None else tensors["sh_down"].shape[1]
        self.max_tokens = max_tokens
        # one workspace for every token count up to max_tokens: its counters
        # sit in a fixed header and return to zero after every call
        self.ws = Workspace(ffn_workspace_bytes_upto(max_tokens, self.H, self.I, self.Is, recipe),
                            tensors["gate"].device)

    def routing_independent(self):
        """The tensors of this layer that do not depend on its routing: the
        router gate and biases, the shared expert and its gate."""
        t = self.t
        keys = ["gate", "router_bias", "expert_bias", "sh_gate", "sh_gate_up", "sh_down", "sh_gate_up_q", "sh_down_q"]
        return [t[k] for k in keys if t.get(k) is not None]

    def forward(self, x, y=None, topk_idx_out=None, topk_w_out=None, counts_out=None, stream=None, ahead=None):
        """ahead: the next MoELayer, whose routing-independent weights this
        forward prefetches into L2 in its expert kernel's tail."""
        T = x.shape[0]
        if ahead is not None:
            set_l2_prefetch(ahead.routing_independent())
        if T > self.max_tokens:
            raise ValueError("more tokens than the workspace was sized for")
        t = self.t
        if self.mx:
            return moe_ffn_forward_mx(x, t["gate"], self.fmt, t["w_gate_up_q"], t["w_down_q"], self.scales,
                                      self.recipe, self.ws, self.I, router_bias=t.get("router_bias"),
                                      expert_bias=t.get("expert_bias"), sh_gate_up_q=t.get("sh_gate_up_q"),
                                      sh_down_q=t.get("sh_down_q"), sh_gate=t.get("sh_gate"), y=y,
                                      topk_idx_out=topk_idx_out, topk_w_out=topk_w_out, counts_out=counts_out,
                                      stream=stream)
        if self.fp4:
            return moe_ffn_forward_fp4(x, t["gate"], t["w_gate_up_q"], t["w_down_q"], self.scales, self.recipe,
                                       self.ws, router_bias=t.get("router_bias"), expert_bias=t.get("expert_bias"),
                                       sh_gate_up=t.get("sh_gate_up"), sh_down=t.get("sh_down"),
                                       sh_gate=t.get("sh_gate"), y=y, topk_idx_out=topk_idx_out,
                                       topk_w_out=topk_w_out, counts_out=counts_out, stream=stream)
        return moe_ffn_forward(x, t["gate"], t["w_gate_up"], t["w_down"], self.recipe, self.ws,
                               router_bias=t.get("router_bias"), expert_bias=t.get("expert_bias"),
                               sh_gate_up=t.get("sh_gate_up"), sh_down=t.get("sh_down"), sh_gate=t.get("sh_gate"),
                               y=y, topk_idx_out=topk_idx_out, topk_w_out=topk_w_out, counts_out=counts_out,
                               stream=stream)
