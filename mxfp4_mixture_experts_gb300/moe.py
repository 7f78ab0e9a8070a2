"""ctypes binding of libmxfp4_moe.so (C ABI: include/mxfp4_moe.h).

Argument marshalling only: every entry point takes PyTorch CUDA tensors,
checks dtype / shape / device, and passes raw device pointers plus the current
CUDA stream to the library. All computation happens in the library's kernels;
there is no fallback: if the library is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxfp4_moe.so")

OK, ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE = range(7)

_lib = None


class MoEError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (code {code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with mxfp4_mixture_experts_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.mxfp4_moe_workspace_size.argtypes = [i32] * 5
    L.mxfp4_moe_workspace_size.restype = sz
    L.mxfp4_moe_workspace_zero_bytes.argtypes = []
    L.mxfp4_moe_workspace_zero_bytes.restype = sz
    L.mxfp4_moe_route.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
    L.mxfp4_moe_route.restype = i32
    L.mxfp4_moe_route_workspace_size.argtypes = [i32, i32, i32]
    L.mxfp4_moe_route_workspace_size.restype = sz
    L.mxfp4_moe_route_ws.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    L.mxfp4_moe_route_ws.restype = i32
    L.mxfp4_moe_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                    vp, vp, vp, sz, i32, vp]
    L.mxfp4_moe_forward.restype = i32
    L.mxfp4_moe_forward_oai.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                        i32, vp, vp, vp, sz, i32, vp]
    L.mxfp4_moe_forward_oai.restype = i32
    L.mxfp4_moe_router.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
    L.mxfp4_moe_router.restype = i32
    L.mxfp4_moe_router_grouped.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    L.mxfp4_moe_router_grouped.restype = i32
    L.mxfp4_moe_forward_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                           i32, i32, vp, vp, vp, sz, i32, vp]
    L.mxfp4_moe_forward_window.restype = i32
    L.mxfp4_moe_encode.argtypes = [vp, i32, i32, i32, vp, vp, vp]
    L.mxfp4_moe_encode.restype = i32
    L.mxfp4_moe_dequant.argtypes = [vp, vp, i32, i32, vp, vp]
    L.mxfp4_moe_dequant.restype = i32
    L.mxfp4_moe_dequant_form.argtypes = [vp, vp, i32, i32, i32, vp, vp]
    L.mxfp4_moe_dequant_form.restype = i32
    L.mxfp4_moe_test_skip_grid_arrival.argtypes = [i32]
    L.mxfp4_moe_test_skip_grid_arrival.restype = None
    L.mxfp4_moe_test_decode_form.argtypes = [i32] * 6
    L.mxfp4_moe_test_decode_form.restype = i32
    L.mxfp4_moe_set_phase_events.argtypes = [vp, i32]
    L.mxfp4_moe_set_phase_events.restype = None
    L.mxfp4_moe_strerror.argtypes = [i32]
    L.mxfp4_moe_strerror.restype = ctypes.c_char_p
    L.mxfp4_moe_version.argtypes = []
    L.mxfp4_moe_version.restype = i32
    _lib = L
    return L


def decode_form(T: int, K: int, I: int, E: int, topk: int, max_smem: int = 232448) -> int:
    """Warps per CTA of the decode form a call of this shape and T runs (7: seven
    consumer warps and a producer), 0 when none fits, -1 for shapes the decode
    path does not take. Host only (227 KB of shared memory per block by default)."""
    return lib().mxfp4_moe_test_decode_form(T, K, I, E, topk, max_smem)


def strerror(code: int) -> str:
    return lib().mxfp4_moe_strerror(int(code)).decode()


def version() -> int:
    return lib().mxfp4_moe_version()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(T: int, K: int, I: int, E: int, topk: int) -> int:
    return int(lib().mxfp4_moe_workspace_size(T, K, I, E, topk))


def workspace_zero_bytes() -> int:
    """Bytes at the start of a workspace that must be zero before first use
    (every call leaves them zero)."""
    return int(lib().mxfp4_moe_workspace_zero_bytes())


def new_workspace(T: int, K: int, I: int, E: int, topk: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (the library requires zeros before first use)."""
    n = workspace_size(T, K, I, E, topk)
    if n == 0:
        raise ValueError("unsupported sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def route(topk_ids: torch.Tensor, E: int, stream=None, many_ctas: bool = False):
    """Stable counting sort of routes by expert -> (count[E], offset[E+1],
    route_list[T*k], status[4]), all int32 CUDA tensors. many_ctas takes
    mxfp4_moe_route_ws (the prefill path's sort, over many CTAs from 8192
    routes on) with scratch allocated here."""
    _need(topk_ids, "topk_ids", torch.int32, 2)
    T, k = topk_ids.shape
    dev = topk_ids.device
    count = torch.empty(E, dtype=torch.int32, device=dev)
    offset = torch.empty(E + 1, dtype=torch.int32, device=dev)
    lst = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    if many_ctas:
        n = int(lib().mxfp4_moe_route_workspace_size(T, k, E))
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        rc = lib().mxfp4_moe_route_ws(_ptr(topk_ids), T, k, E, _ptr(count), _ptr(offset),
                                      _ptr(lst), _ptr(status), _ptr(ws), n, _stream(stream))
        if rc:
            raise MoEError(rc, "mxfp4_moe_route_ws")
    else:
        rc = lib().mxfp4_moe_route(_ptr(topk_ids), T, k, E, _ptr(count), _ptr(offset),
                                   _ptr(lst), _ptr(status), _stream(stream))
        if rc:
            raise MoEError(rc, "mxfp4_moe_route")
    return count, offset, lst[:T * k], status


def forward(hidden: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
            w13: torch.Tensor, s13: torch.Tensor, w2: torch.Tensor, s2: torch.Tensor,
            out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
            status: Optional[torch.Tensor] = None, path: int = 0, stream=None) -> torch.Tensor:
    """y[T, K] bf16 = sum_j w_tj * W2[e] (silu(W_gate[e] x_t) * (W_up[e] x_t))."""
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_weights, "topk_weights", torch.float32, 2)
    for n, t in (("w13", w13), ("s13", s13), ("w2", w2), ("s2", s2)):
        _need(t, n, torch.uint8, 3)
    T, K = hidden.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    k = topk_ids.shape[1]
    if tuple(topk_ids.shape) != (T, k) or tuple(topk_weights.shape) != (T, k):
        raise ValueError("topk_ids / topk_weights must be [T, topk]")
    if tuple(w13.shape) != (E, 2 * I, K // 2) or tuple(s13.shape) != (E, 2 * I, K // 32):
        raise ValueError("w13 / s13 shapes must be [E, 2I, K/2] / [E, 2I, K/32]")
    if tuple(w2.shape) != (E, K, I // 2) or tuple(s2.shape) != (E, K, I // 32):
        raise ValueError("w2 / s2 shapes must be [E, K, I/2] / [E, K, I/32]")
    if out is None:
        out = torch.empty(T, K, dtype=torch.bfloat16, device=hidden.device)
    else:
        _need(out, "out", torch.bfloat16, 2)
    if workspace is None:
        workspace = new_workspace(T, K, I, E, k, hidden.device)
    rc = lib().mxfp4_moe_forward(
        _ptr(hidden), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13), _ptr(s13), _ptr(w2),
        _ptr(s2), T, K, I, E, k, _ptr(out), _ptr(status), _ptr(workspace),
        workspace.numel() * workspace.element_size(), path, _stream(stream))
    if rc:
        raise MoEError(rc, "mxfp4_moe_forward")
    return out


def forward_window(hidden: torch.Tensor, topk_ids: torch.Tensor,
                   topk_weights: Optional[torch.Tensor], w13: torch.Tensor, s13: torch.Tensor,
                   w2: torch.Tensor, s2: torch.Tensor, expert_base: int = 0,
                   per_route: bool = False, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                   path: int = 0, stream=None) -> torch.Tensor:
    """The layer over the experts expert_base .. expert_base + E - 1 held by
    w13/s13/w2/s2 (other ids skipped): y [T, K] of the window's routes, or with
    per_route each route's unweighted w2 output [T * topk, K]."""
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    if topk_weights is not None:
        _need(topk_weights, "topk_weights", torch.float32, 2)
    elif not per_route:
        raise ValueError("topk_weights are needed unless per_route")
    for n, t in (("w13", w13), ("s13", s13), ("w2", w2), ("s2", s2)):
        _need(t, n, torch.uint8, 3)
    T, K = hidden.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    k = topk_ids.shape[1]
    rows = T * k if per_route else T
    if out is None:
        out = torch.empty(rows, K, dtype=torch.bfloat16, device=hidden.device)
    else:
        _need(out, "out", torch.bfloat16, 2)
        if tuple(out.shape) != (rows, K):
            raise ValueError(f"out must be [{rows}, {K}]")
    if workspace is None:
        workspace = new_workspace(T, K, I, E, k, hidden.device)
    rc = lib().mxfp4_moe_forward_window(
        _ptr(hidden), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13), _ptr(s13), _ptr(w2),
        _ptr(s2), T, K, I, E, k, int(expert_base), int(bool(per_route)), _ptr(out), _ptr(status),
        _ptr(workspace), workspace.numel() * workspace.element_size(), path, _stream(stream))
    if rc:
        raise MoEError(rc, "mxfp4_moe_forward_window")
    return out


def forward_oai(hidden: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                w13: torch.Tensor, s13: torch.Tensor, b13: torch.Tensor,
                w2: torch.Tensor, s2: torch.Tensor, b2: torch.Tensor,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, path: int = 0, stream=None) -> torch.Tensor:
    """The gpt-oss form: w13 rows interleaved (row 2i gate i, row 2i + 1 up i),
    f32 biases b13 [E, 2I] (same row order) and b2 [E, K], SwiGLU-OAI;
    y[T, K] bf16 = sum_j w_tj * (W2[e] h + b2[e]). Paths as forward()."""
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_weights, "topk_weights", torch.float32, 2)
    for n, t in (("w13", w13), ("s13", s13), ("w2", w2), ("s2", s2)):
        _need(t, n, torch.uint8, 3)
    _need(b13, "b13", torch.float32, 2)
    _need(b2, "b2", torch.float32, 2)
    T, K = hidden.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    k = topk_ids.shape[1]
    if tuple(topk_ids.shape) != (T, k) or tuple(topk_weights.shape) != (T, k):
        raise ValueError("topk_ids / topk_weights must be [T, topk]")
    if tuple(w13.shape) != (E, 2 * I, K // 2) or tuple(s13.shape) != (E, 2 * I, K // 32):
        raise ValueError("w13 / s13 shapes must be [E, 2I, K/2] / [E, 2I, K/32]")
    if tuple(w2.shape) != (E, K, I // 2) or tuple(s2.shape) != (E, K, I // 32):
        raise ValueError("w2 / s2 shapes must be [E, K, I/2] / [E, K, I/32]")
    if tuple(b13.shape) != (E, 2 * I) or tuple(b2.shape) != (E, K):
        raise ValueError("b13 / b2 shapes must be [E, 2I] / [E, K]")
    if out is None:
        out = torch.empty(T, K, dtype=torch.bfloat16, device=hidden.device)
    else:
        _need(out, "out", torch.bfloat16, 2)
    if workspace is None:
        workspace = new_workspace(T, K, I, E, k, hidden.device)
    rc = lib().mxfp4_moe_forward_oai(
        _ptr(hidden), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13), _ptr(s13), _ptr(b13),
        _ptr(w2), _ptr(s2), _ptr(b2), T, K, I, E, k, _ptr(out), _ptr(status), _ptr(workspace),
        workspace.numel() * workspace.element_size(), path, _stream(stream))
    if rc:
        raise MoEError(rc, "mxfp4_moe_forward_oai")
    return out


SCORING = {"softmax_topk": 0, "sigmoid_renorm": 1}


def _router_args(logits, topk, scoring, bias, topk_ids, topk_weights):
    _need(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    if bias is not None:
        _need(bias, "bias", torch.float32, 1)
        if bias.shape[0] != E:
            raise ValueError("bias must be [E]")
    if scoring not in SCORING:
        raise ValueError(f"scoring must be one of {sorted(SCORING)}")
    if topk_ids is None:
        topk_ids = torch.empty(T, topk, dtype=torch.int32, device=logits.device)
    if topk_weights is None:
        topk_weights = torch.empty(T, topk, dtype=torch.float32, device=logits.device)
    return T, E, topk_ids, topk_weights


def router(logits: torch.Tensor, topk: int, scoring: str = "softmax_topk",
           bias: Optional[torch.Tensor] = None, topk_ids: Optional[torch.Tensor] = None,
           topk_weights: Optional[torch.Tensor] = None, stream=None):
    """Top-k experts of fp32 logits [T, E] (+ bias [E]) and their weights:
    int32 [T, k] ids (descending x = logit + bias, ties to the lower index)
    and fp32 [T, k] weights (softmax over the chosen, or renormalised sigmoid)."""
    T, E, topk_ids, topk_weights = _router_args(logits, topk, scoring, bias, topk_ids,
                                                topk_weights)
    rc = lib().mxfp4_moe_router(_ptr(logits), _ptr(bias), T, E, topk, SCORING[scoring],
                                _ptr(topk_ids), _ptr(topk_weights), _stream(stream))
    if rc:
        raise MoEError(rc, "mxfp4_moe_router")
    return topk_ids, topk_weights


def router_grouped(logits: torch.Tensor, topk: int, scoring: str = "sigmoid_renorm",
                   bias: Optional[torch.Tensor] = None, n_group: int = 1, topk_group: int = 1,
                   bias_in_weights: bool = True, topk_ids: Optional[torch.Tensor] = None,
                   topk_weights: Optional[torch.Tensor] = None, stream=None):
    """``router`` with grouped top-k (n_group groups of consecutive experts
    scored by their largest x; the experts of the topk_group best groups stay
    eligible) and, with bias_in_weights=False, a bias that steers the choice
    only (weights from the unbiased logits)."""
    T, E, topk_ids, topk_weights = _router_args(logits, topk, scoring, bias, topk_ids,
                                                topk_weights)
    rc = lib().mxfp4_moe_router_grouped(_ptr(logits), _ptr(bias), T, E, topk, SCORING[scoring],
                                        n_group, topk_group, int(bool(bias_in_weights)),
                                        _ptr(topk_ids), _ptr(topk_weights), _stream(stream))
    if rc:
        raise MoEError(rc, "mxfp4_moe_router_grouped")
    return topk_ids, topk_weights


RULES = {"ocp": 0, "quark": 1}


def encode(x: torch.Tensor, rule: str = "ocp", stream=None):
    """bf16 [rows, cols] -> (packed uint8 [rows, cols/2], E8M0 scales uint8
    [rows, cols/32]); rule "ocp" (floor(log2 amax) - 2) or "quark" (raised by
    one when amax / 2^X >= 7)."""
    _need(x, "x", torch.bfloat16, 2)
    if rule not in RULES:
        raise ValueError(f"rule must be one of {sorted(RULES)}")
    rows, cols = x.shape
    packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
    scale = torch.empty(rows, cols // 32, dtype=torch.uint8, device=x.device)
    rc = lib().mxfp4_moe_encode(_ptr(x), rows, cols, RULES[rule], _ptr(packed), _ptr(scale),
                                _stream(stream))
    if rc:
        raise MoEError(rc, "mxfp4_moe_encode")
    return packed, scale


DEQUANT_FORMS = {"decode": 1, "prefill": 2}


def dequant(packed: torch.Tensor, scale: torch.Tensor, form: str = "decode",
            stream=None) -> torch.Tensor:
    """Packed rows [N, C/2] + scales [N, C/32] -> bf16 [N, C], through the
    weight decode of the decode kernels (form "decode") or of the prefill
    GEMM (form "prefill")."""
    _need(packed, "packed", torch.uint8, 2)
    _need(scale, "scale", torch.uint8, 2)
    if form not in DEQUANT_FORMS:
        raise ValueError(f"form must be one of {sorted(DEQUANT_FORMS)}")
    N, half = packed.shape
    C = 2 * half
    if tuple(scale.shape) != (N, C // 32):
        raise ValueError("scale must be [rows, cols/32]")
    out = torch.empty(N, C, dtype=torch.bfloat16, device=packed.device)
    rc = lib().mxfp4_moe_dequant_form(_ptr(packed), _ptr(scale), N, C, DEQUANT_FORMS[form],
                                      _ptr(out), _stream(stream))
    if rc:
        raise MoEError(rc, "mxfp4_moe_dequant_form")
    return out


def set_phase_events(events) -> None:
    """Profiling hook: list of torch.cuda.Event (>= 3) recorded around each
    kernel of later forward calls, or None to disable."""
    L = lib()
    if events is None:
        L.mxfp4_moe_set_phase_events(None, 0)
        set_phase_events._keep = None
        return
    for e in events:
        if e.cuda_event == 0:     # torch creates the CUDA event on first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    set_phase_events._keep = arr   # the library keeps the pointer
    L.mxfp4_moe_set_phase_events(ctypes.cast(arr, ctypes.c_void_p), len(events))
