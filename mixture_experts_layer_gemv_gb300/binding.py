"""Thin Python binding of libmoe_gb300.so (include/moe.h), same entry-point names.

Argument marshalling only: torch tensors supply device pointers and the current
CUDA stream; every step of the layer runs in the library's CUDA kernels. There is
no fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, Optional

import torch

from .synth import MoEConfig

PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_GB300_LIB: another build of the library (the MOE_DEBUG build, for instance)
LIB_PATH = os.environ.get("MOE_GB300_LIB") or os.path.join(PKG, "libmoe_gb300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "moe.h")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED_SHAPE",
                -3: "MOE_ERR_WORKSPACE", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE_TIMEOUT"}
STAGES = ("route", "permute", "gate_up", "down", "combine")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}: {text}")
        self.status = status


class moe_config_t(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("moe_inter", ctypes.c_int32), ("n_routed", ctypes.c_int32),
                ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float)]


_WEIGHT_FIELDS = ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down", "ws_gate", "ws_up", "ws_down",
                  "ss_gate", "ss_up", "ss_down", "w_router", "router_bias")


class moe_weights_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


class moe_weights_mx_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


class moe_stage_events_t(ctypes.Structure):
    _fields_ = [("start", ctypes.c_void_p * 5), ("stop", ctypes.c_void_p * 5)]


_P, _I32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_workspace_size": (_SZ, [_P, _I32]),
    "moe_workspace_init": (ctypes.c_int, [_P, _SZ, _P]),
    "moe_read_device_status": (ctypes.c_int, [_P, _P]),
    "moe_debug_set": (ctypes.c_int, [_P, _SZ, ctypes.c_uint32, _P]),
    "moe_backward_workspace_size": (_SZ, [_P, _I32]),
    "moe_backward": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                    _P]),
    "moe_backward_profiled": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                             _P, _SZ, _P, _P]),
    "moe_quant_act": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P]),
    "moe_rmsnorm": (ctypes.c_int, [_P, _I32, _I32, _P, ctypes.c_float, _P, _P]),
    "moe_route_rmsnorm": (ctypes.c_int, [_P, _P, _I32, _P, ctypes.c_float, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_rmsnorm": (ctypes.c_int, [_P, _P, _I32, _P, ctypes.c_float, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_rmsnorm_profiled": (ctypes.c_int, [_P, _P, _I32, _P, ctypes.c_float, _P, _P, _P, _P, _SZ, _P,
                                                    _P]),
    "moe_route": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_route_noalloc": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P]),
    "moe_permute": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_ffn": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_combine": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P, _P]),
    "moe_forward": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_profiled": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "moe_forward_trace": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _SZ, _P, _P]),
    "moe_workspace_size_mx": (_SZ, [_P, _I32]),
    "moe_quant_act_mx": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P]),
    "moe_forward_mx": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_mx_profiled": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P, _P]),
}

_lib = None


def declared_symbols():
    """Entry points declared in include/moe.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*[\w\s\*]*?\b(moe_\w+)\s*\(", text, re.M)))


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(python -m mixture_experts_layer_gemv_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status, status_string(status))


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def config_struct(cfg: MoEConfig) -> moe_config_t:
    return moe_config_t(cfg.hidden, cfg.moe_inter, cfg.n_routed, cfg.n_group, cfg.topk_group, cfg.top_k,
                        cfg.n_shared, float(cfg.routed_scaling_factor))


def weights_struct(weights: Dict[str, Optional[torch.Tensor]]) -> moe_weights_t:
    return moe_weights_t(*[_ptr(weights.get(n)) for n in _WEIGHT_FIELDS])


# ----------------------------------------------------------------- workspace
def moe_workspace_size(cfg: MoEConfig, max_tokens: int) -> int:
    c = config_struct(cfg)
    return int(lib().moe_workspace_size(ctypes.byref(c), int(max_tokens)))


def moe_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check("moe_workspace_init", lib().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def alloc_workspace(cfg: MoEConfig, max_tokens: int, device="cuda") -> torch.Tensor:
    n = moe_workspace_size(cfg, max_tokens)
    if n == 0:
        raise MoeError("moe_workspace_size", -2, "invalid config")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


INJECT_SKIP_GATEUP_LOADS = 1


def moe_debug_set(ws: torch.Tensor, inject: int = 0, stream=None) -> None:
    """Failure-detection test hook: the fault-injection bits for the calls that follow on
    ws (see moe.h); 0 clears them."""
    _check("moe_debug_set", lib().moe_debug_set(_ptr(ws), ws.numel() * ws.element_size(), int(inject),
                                                _stream(stream)))


def moe_read_device_status(ws: torch.Tensor, stream=None) -> int:
    return int(lib().moe_read_device_status(_ptr(ws), _stream(stream)))


# ------------------------------------------------------------------- stages
def moe_quant_act(x: torch.Tensor, xq: torch.Tensor, xs: torch.Tensor, stream=None) -> None:
    T, H = x.shape
    _check("moe_quant_act", lib().moe_quant_act(_ptr(x), T, H, _ptr(xq), _ptr(xs), _stream(stream)))


def moe_rmsnorm(h: torch.Tensor, gamma: torch.Tensor, eps: float, x_out: torch.Tensor, stream=None) -> None:
    """Stage M: x_out = bf16(h / sqrt(mean(h^2) + eps) * gamma) per row."""
    T, H = h.shape
    _check("moe_rmsnorm", lib().moe_rmsnorm(_ptr(h), T, H, _ptr(gamma), float(eps), _ptr(x_out), _stream(stream)))


def moe_route_rmsnorm(cfg, h, gamma, eps, w_router, router_bias, topk_ids, topk_w, ws, stream=None) -> None:
    c = config_struct(cfg)
    _check("moe_route_rmsnorm", lib().moe_route_rmsnorm(ctypes.byref(c), _ptr(h), h.shape[0], _ptr(gamma),
                                                        float(eps), _ptr(w_router), _ptr(router_bias),
                                                        _ptr(topk_ids), _ptr(topk_w), _ptr(ws), ws.numel(),
                                                        _stream(stream)))


def moe_route(cfg, x, w_router, router_bias, topk_ids, topk_w, ws, stream=None) -> None:
    c = config_struct(cfg)
    _check("moe_route", lib().moe_route(ctypes.byref(c), _ptr(x), x.shape[0], _ptr(w_router), _ptr(router_bias),
                                        _ptr(topk_ids), _ptr(topk_w), _ptr(ws), ws.numel(), _stream(stream)))


def moe_route_noalloc(cfg, x, w_router, router_bias, topk_ids, topk_w, stream=None) -> None:
    """moe_route for callers that cannot allocate: no workspace argument; the library's
    fixed internal scratch (T <= 64, n_routed <= 256, hidden <= 8192) is used instead.
    Calls that overlap on the GPU share that scratch and must be serialised."""
    c = config_struct(cfg)
    _check("moe_route_noalloc", lib().moe_route_noalloc(ctypes.byref(c), _ptr(x), x.shape[0], _ptr(w_router),
                                                        _ptr(router_bias), _ptr(topk_ids), _ptr(topk_w),
                                                        _stream(stream)))


def moe_permute(cfg, topk_ids, expert_offsets, perm_src, inv_pos, ws, stream=None) -> None:
    c = config_struct(cfg)
    _check("moe_permute", lib().moe_permute(ctypes.byref(c), _ptr(topk_ids), topk_ids.shape[0],
                                            _ptr(expert_offsets), _ptr(perm_src), _ptr(inv_pos), _ptr(ws),
                                            ws.numel(), _stream(stream)))


def moe_expert_ffn(cfg, x, weights, expert_offsets, perm_src, topk_w, y_perm, y_shared, ws, stream=None) -> None:
    c = config_struct(cfg)
    W = weights_struct(weights)
    _check("moe_expert_ffn", lib().moe_expert_ffn(ctypes.byref(c), _ptr(x), x.shape[0], ctypes.byref(W),
                                                  _ptr(expert_offsets), _ptr(perm_src), _ptr(topk_w),
                                                  _ptr(y_perm), _ptr(y_shared), _ptr(ws), ws.numel(),
                                                  _stream(stream)))


def moe_combine(cfg, y_perm, inv_pos, y_shared, residual, out, stream=None) -> None:
    c = config_struct(cfg)
    _check("moe_combine", lib().moe_combine(ctypes.byref(c), _ptr(y_perm), _ptr(inv_pos), _ptr(y_shared),
                                            _ptr(residual), out.shape[0], _ptr(out), _stream(stream)))


def moe_forward(cfg, x, weights, out, residual=None, topk_ids_out=None, ws=None, stream=None,
                events: Optional[Dict[str, tuple]] = None) -> None:
    """out[T, H] (bf16) = MoE layer(x); ws from alloc_workspace(cfg, >= T).

    events: optional {stage name: (start torch.cuda.Event, stop torch.cuda.Event)}
    recorded around that stage's kernels.
    """
    c = config_struct(cfg)
    W = weights_struct(weights)
    if events:
        ev = _events_struct(events)
        st = lib().moe_forward_profiled(ctypes.byref(c), _ptr(x), x.shape[0], ctypes.byref(W), _ptr(residual),
                                        _ptr(out), _ptr(topk_ids_out), _ptr(ws), ws.numel(), _stream(stream),
                                        ctypes.byref(ev))
        _check("moe_forward_profiled", st)
        return
    _check("moe_forward", lib().moe_forward(ctypes.byref(c), _ptr(x), x.shape[0], ctypes.byref(W), _ptr(residual),
                                            _ptr(out), _ptr(topk_ids_out), _ptr(ws), ws.numel(), _stream(stream)))


TRACE_CTAS = 512
TRACE_WORDS = 4 * TRACE_CTAS * 4
TRACE_KERNELS = ("route", "gate_up", "down", "combine")
TRACE_EVENTS = ("start", "wait_done", "first_data", "done")


def moe_forward_trace(cfg, x, weights, out, trace, residual=None, ws=None, stream=None) -> None:
    """moe_forward that also writes per-CTA global-timer stamps into trace (int64 device
    tensor of TRACE_WORDS): trace.view(4, TRACE_CTAS, 4)[kernel, cta, event] in ns."""
    c = config_struct(cfg)
    W = weights_struct(weights)
    _check("moe_forward_trace", lib().moe_forward_trace(ctypes.byref(c), _ptr(x), x.shape[0], ctypes.byref(W),
                                                        _ptr(residual), _ptr(out), _ptr(ws), ws.numel(),
                                                        _stream(stream), _ptr(trace)))


def _events_struct(events):
    ev = moe_stage_events_t()
    for name, (a, b) in events.items():
        i = STAGES.index(name)
        ev.start[i] = a.cuda_event
        ev.stop[i] = b.cuda_event
    return ev


def moe_forward_rmsnorm(cfg, h, gamma, eps, weights, out, topk_ids_out=None, ws=None, stream=None,
                        events: Optional[Dict[str, tuple]] = None) -> None:
    """out[T, H] = h + MoE layer(RMSNorm(h) * gamma); ws from alloc_workspace(cfg, >= T)."""
    c = config_struct(cfg)
    W = weights_struct(weights)
    if events:
        ev = _events_struct(events)
        st = lib().moe_forward_rmsnorm_profiled(ctypes.byref(c), _ptr(h), h.shape[0], _ptr(gamma), float(eps),
                                                ctypes.byref(W), _ptr(out), _ptr(topk_ids_out), _ptr(ws),
                                                ws.numel(), _stream(stream), ctypes.byref(ev))
        _check("moe_forward_rmsnorm_profiled", st)
        return
    _check("moe_forward_rmsnorm", lib().moe_forward_rmsnorm(ctypes.byref(c), _ptr(h), h.shape[0], _ptr(gamma),
                                                            float(eps), ctypes.byref(W), _ptr(out),
                                                            _ptr(topk_ids_out), _ptr(ws), ws.numel(),
                                                            _stream(stream)))


# ------------------------------------------------------------ MXFP8 variant
def weights_mx_struct(weights: Dict[str, Optional[torch.Tensor]]) -> moe_weights_mx_t:
    return moe_weights_mx_t(*[_ptr(weights.get(n)) for n in _WEIGHT_FIELDS])


def moe_workspace_size_mx(cfg: MoEConfig, max_tokens: int) -> int:
    c = config_struct(cfg)
    return int(lib().moe_workspace_size_mx(ctypes.byref(c), int(max_tokens)))


def alloc_workspace_mx(cfg: MoEConfig, max_tokens: int, device="cuda") -> torch.Tensor:
    n = moe_workspace_size_mx(cfg, max_tokens)
    if n == 0:
        raise MoeError("moe_workspace_size_mx", -2, "config not supported by the MXFP8 variant")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


def moe_quant_act_mx(x: torch.Tensor, xq: torch.Tensor, xs8: torch.Tensor, stream=None) -> None:
    T, H = x.shape
    _check("moe_quant_act_mx", lib().moe_quant_act_mx(_ptr(x), T, H, _ptr(xq), _ptr(xs8), _stream(stream)))


def moe_forward_mx(cfg, x, weights, out, residual=None, topk_ids_out=None, ws=None, stream=None,
                   events: Optional[Dict[str, tuple]] = None) -> None:
    """out[T, H] = MoE layer(x) with MXFP8 experts (weights from synth.make_weights_mx)."""
    c = config_struct(cfg)
    W = weights_mx_struct(weights)
    if events:
        st = lib().moe_forward_mx_profiled(ctypes.byref(c), _ptr(x), x.shape[0], ctypes.byref(W), _ptr(residual),
                                           _ptr(out), _ptr(topk_ids_out), _ptr(ws), ws.numel(), _stream(stream),
                                           ctypes.byref(_events_struct(events)))
        _check("moe_forward_mx_profiled", st)
        return
    _check("moe_forward_mx", lib().moe_forward_mx(ctypes.byref(c), _ptr(x), x.shape[0], ctypes.byref(W),
                                                  _ptr(residual), _ptr(out), _ptr(topk_ids_out), _ptr(ws),
                                                  ws.numel(), _stream(stream)))


def forward_mx(cfg: MoEConfig, x: torch.Tensor, weights, residual=None, ws=None, return_ids=False):
    T = x.shape[0]
    ws = alloc_workspace_mx(cfg, T, x.device) if ws is None else ws
    out = torch.empty_like(x)
    ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device=x.device) if return_ids else None
    moe_forward_mx(cfg, x, weights, out, residual, ids, ws)
    return (out, ids) if return_ids else out


def forward(cfg: MoEConfig, x: torch.Tensor, weights, residual=None, ws=None, return_ids=False):
    """Convenience: allocate out (and ws if not given) and run moe_forward."""
    T = x.shape[0]
    ws = alloc_workspace(cfg, T, x.device) if ws is None else ws
    out = torch.empty_like(x)
    ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device=x.device) if return_ids else None
    moe_forward(cfg, x, weights, out, residual, ids, ws)
    return (out, ids) if return_ids else out


def moe_backward_workspace_size(cfg: MoEConfig, max_tokens: int) -> int:
    c = config_struct(cfg)
    return lib().moe_backward_workspace_size(ctypes.byref(c), max_tokens)


def alloc_workspace_backward(cfg: MoEConfig, max_tokens: int, device="cuda") -> torch.Tensor:
    n = moe_backward_workspace_size(cfg, max_tokens)
    if n == 0:
        raise MoeError("moe_backward_workspace_size", -2, "config not supported by the backward")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


def moe_backward(cfg, x, weights, topk_ids, topk_w, dout, grads: Dict[str, torch.Tensor], ws, stream=None,
                 events: Optional[Dict[str, tuple]] = None) -> None:
    """Fill grads (fp32 tensors: dx, dw_gate, dw_up, dw_down, dws_gate, dws_up, dws_down,
    dw_router, dbias) with the layer's gradients for output gradient dout. events: as
    for moe_forward, in the backward's slots (see moe.h, moe_backward_profiled)."""
    c = config_struct(cfg)
    W = weights_struct(weights)
    g = grads
    args = [ctypes.byref(c), _ptr(x), x.shape[0], ctypes.byref(W), _ptr(topk_ids), _ptr(topk_w), _ptr(dout),
            _ptr(g["dx"]), _ptr(g["dw_gate"]), _ptr(g["dw_up"]), _ptr(g["dw_down"]), _ptr(g.get("dws_gate")),
            _ptr(g.get("dws_up")), _ptr(g.get("dws_down")), _ptr(g["dw_router"]), _ptr(g.get("dbias")), _ptr(ws),
            ws.numel(), _stream(stream)]
    if events:
        _check("moe_backward_profiled", lib().moe_backward_profiled(*args, ctypes.byref(_events_struct(events))))
    else:
        _check("moe_backward", lib().moe_backward(*args))


def alloc_grads(cfg: MoEConfig, T: int, device="cuda", bias=True) -> Dict[str, torch.Tensor]:
    H, I, E, Is = cfg.hidden, cfg.moe_inter, cfg.n_routed, cfg.shared_inter
    f = dict(dtype=torch.float32, device=device)
    g = {"dx": torch.empty((T, H), **f), "dw_gate": torch.empty((E, I, H), **f), "dw_up": torch.empty((E, I, H), **f),
         "dw_down": torch.empty((E, H, I), **f), "dw_router": torch.empty((E, H), **f)}
    if Is > 0:
        g.update(dws_gate=torch.empty((Is, H), **f), dws_up=torch.empty((Is, H), **f),
                 dws_down=torch.empty((H, Is), **f))
    if bias:
        g["dbias"] = torch.empty((E,), **f)
    return g


def backward(cfg: MoEConfig, x: torch.Tensor, weights, topk_ids, topk_w, dout, ws=None) -> Dict[str, torch.Tensor]:
    """Convenience: allocate the gradients (and ws if not given) and run moe_backward."""
    T = x.shape[0]
    ws = alloc_workspace_backward(cfg, T, x.device) if ws is None else ws
    g = alloc_grads(cfg, T, x.device)
    moe_backward(cfg, x, weights, topk_ids, topk_w, dout, g, ws)
    return g
