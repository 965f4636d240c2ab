"""ctypes front end of the fp64 CPU oracle (moe_oracle.cpp).

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg import this package. The product path never does: the CUDA library
fails loudly when its extension is missing instead of falling back here.

Every function takes and returns numpy arrays on the host. bf16 activations are
passed as their raw 16-bit patterns (uint16), E4M3 weights as uint8 codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "moe_oracle.cpp")
LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libmoe_oracle.so next to its source (g++ -O3 -fopenmp)."""
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SRC):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O3", "-fopenmp", "-shared", "-fPIC", SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32),
        ("moe_inter", ctypes.c_int32),
        ("n_routed", ctypes.c_int32),
        ("n_group", ctypes.c_int32),
        ("topk_group", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("n_shared", ctypes.c_int32),
        ("act_quant", ctypes.c_int32),
        ("routed_scaling_factor", ctypes.c_double),
    ]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
        "ws_gate", "ws_up", "ws_down", "ss_gate", "ss_up", "ss_down")]


_P = ctypes.c_void_p


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB_PATH)
            lib.orc_e4m3_decode.restype = ctypes.c_double
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
            lib.orc_quant_rows.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P]
            lib.orc_round_bf16.argtypes = [_P, ctypes.c_int, _P]
            lib.orc_rmsnorm.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_double, _P, _P]
            lib.orc_router_logits.argtypes = [_P, _P, ctypes.c_int, _P, _P, _P]
            lib.orc_topk.argtypes = [_P, _P, ctypes.c_int, _P, _P, _P, _P]
            lib.orc_permute.argtypes = [_P, _P, ctypes.c_int, _P, _P, _P]
            lib.orc_expert_row.argtypes = [_P, _P, _P, ctypes.c_int, ctypes.c_double, _P, _P]
            lib.orc_shared_row.argtypes = [_P, _P, _P, _P]
            lib.orc_forward_tokens.argtypes = [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P]
            lib.orc_e8m0_decode.restype = ctypes.c_double
            lib.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
            lib.orc_quant_rows_mx.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P]
            lib.orc_forward_tokens_mx.argtypes = [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P]
            lib.orc_forward_fixed_ids_d.argtypes = [_P, _P, _P, _P, _P, ctypes.c_int, _P, _P]
            lib.orc_backward_d.argtypes = [_P, _P, _P, _P, _P, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P,
                                           _P, _P, _P]
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _np(t, dtype):
    """torch tensor / numpy array -> contiguous host numpy array of dtype."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        import torch
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        t = t.contiguous().numpy()
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        if dtype in (np.uint16, np.uint8):  # raw bit patterns: reinterpret, never convert
            assert a.dtype.itemsize == np.dtype(dtype).itemsize, (a.dtype, dtype)
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return np.ascontiguousarray(a)


def _cfg(cfg, act_quant=True):
    return _Cfg(cfg.hidden, cfg.moe_inter, cfg.n_routed, cfg.n_group, cfg.topk_group, cfg.top_k,
                cfg.n_shared, 1 if act_quant else 0, float(cfg.routed_scaling_factor))


class Weights:
    """Host copies of one layer's weights (same keys as synth.make_weights)."""

    KEYS = ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
            "ws_gate", "ws_up", "ws_down", "ss_gate", "ss_up", "ss_down")

    def __init__(self, weights: dict):
        self.arrays = {}
        for k in self.KEYS:
            v = weights.get(k)
            self.arrays[k] = _np(v, np.uint8 if k.startswith("w") else np.float32)
        self.struct = _Weights(*[_ptr(self.arrays[k]) for k in
                                 ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
                                  "ws_gate", "ws_up", "ws_down", "ss_gate", "ss_up", "ss_down")])


class WeightsMX:
    """Host copies of one layer's MXFP8 weights (same keys as synth.make_weights_mx):
    E4M3 codes and E8M0 scale bytes per (row, 32 consecutive K)."""

    KEYS = Weights.KEYS

    def __init__(self, weights: dict):
        self.arrays = {k: _np(weights.get(k), np.uint8) for k in self.KEYS}
        self.struct = _Weights(*[_ptr(self.arrays[k]) for k in self.KEYS])


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e4m3_decode(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.array([lib.orc_e4m3_encode(float(x)) for x in v.ravel()], dtype=np.uint8).reshape(v.shape)


def quant_rows(v) -> tuple:
    """Per (row, 128-column block) FP8 quantisation: (codes uint8 [R,N], scales f64 [R,N/128])."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    R, N = v.shape
    assert N % 128 == 0
    q = np.empty((R, N), np.uint8)
    s = np.empty((R, N // 128), np.float64)
    lib.orc_quant_rows(_ptr(v), R, N, _ptr(q), _ptr(s))
    return q, s


def round_bf16(values) -> np.ndarray:
    """fp64 values -> bf16 bit patterns (uint16), rounded once to nearest, ties to even."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64))
    out = np.empty(v.shape, np.uint16)
    lib.orc_round_bf16(_ptr(v), v.size, _ptr(out))
    return out


def rmsnorm(h_bf16, gamma_bf16, eps: float, return_exact=False):
    """Stage M: x = h / sqrt(mean(h^2) + eps) * gamma per row, rounded once to bf16.

    -> x as bf16 bit patterns uint16 [T, H] (and the fp64 values before rounding)."""
    lib = _load()
    h = _np(h_bf16, np.uint16)
    g = _np(gamma_bf16, np.uint16).reshape(-1)
    T, H = h.shape
    assert g.shape == (H,)
    x = np.empty((T, H), np.uint16)
    ex = np.empty((T, H), np.float64)
    lib.orc_rmsnorm(_ptr(h), T, H, _ptr(g), float(eps), _ptr(x), _ptr(ex))
    return (x, ex) if return_exact else x


def e8m0_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e8m0_decode(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def quant_rows_mx(v) -> tuple:
    """Per (row, 32-column block) MXFP8 quantisation: (codes uint8 [R,N], E8M0 scales uint8 [R,N/32])."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    R, N = v.shape
    assert N % 32 == 0
    q = np.empty((R, N), np.uint8)
    s = np.empty((R, N // 32), np.uint8)
    lib.orc_quant_rows_mx(_ptr(v), R, N, _ptr(q), _ptr(s))
    return q, s


def router_logits(cfg, x_bf16, w_router, bias=None) -> np.ndarray:
    lib = _load()
    x = _np(x_bf16, np.uint16)
    wr = _np(w_router, np.float32)
    b = _np(bias, np.float32)
    T = x.shape[0]
    out = np.empty((T, cfg.n_routed), np.float64)
    c = _cfg(cfg)
    lib.orc_router_logits(ctypes.byref(c), _ptr(x), T, _ptr(wr), _ptr(b), _ptr(out))
    return out


def topk(cfg, logits):
    """-> ids int32 [T,k], w f64 [T,k], probs f64 [T,E], margin f64 [T]."""
    lib = _load()
    lg = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    T = lg.shape[0]
    ids = np.empty((T, cfg.top_k), np.int32)
    w = np.empty((T, cfg.top_k), np.float64)
    p = np.empty((T, cfg.n_routed), np.float64)
    m = np.empty((T,), np.float64)
    c = _cfg(cfg)
    lib.orc_topk(ctypes.byref(c), _ptr(lg), T, _ptr(ids), _ptr(w), _ptr(p), _ptr(m))
    return ids, w, p, m


def route(cfg, x_bf16, w_router, bias=None):
    """Router + top-k: ids, w, probs, margin."""
    return topk(cfg, router_logits(cfg, x_bf16, w_router, bias))


def permute(cfg, ids):
    """-> expert_offsets [E+1], perm_src [T*k], inv_pos [T*k] (int32)."""
    lib = _load()
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    T = ids.shape[0]
    n = T * cfg.top_k
    off = np.empty((cfg.n_routed + 1,), np.int32)
    ps = np.empty((n,), np.int32)
    ip = np.empty((n,), np.int32)
    c = _cfg(cfg)
    lib.orc_permute(ctypes.byref(c), _ptr(ids), T, _ptr(off), _ptr(ps), _ptr(ip))
    return off, ps, ip


def expert_row(cfg, weights: Weights, x_row_bf16, expert: int, w: float, act_quant=True):
    """y[H] = w * expert(xhat) for one token row; also returns the expert's intermediate ahat[I]."""
    lib = _load()
    x = _np(x_row_bf16, np.uint16).reshape(-1)
    y = np.empty((cfg.hidden,), np.float64)
    a = np.empty((cfg.moe_inter,), np.float64)
    c = _cfg(cfg, act_quant)
    lib.orc_expert_row(ctypes.byref(c), ctypes.byref(weights.struct), _ptr(x), int(expert), float(w),
                       _ptr(y), _ptr(a))
    return y, a


def shared_row(cfg, weights: Weights, x_row_bf16, act_quant=True):
    lib = _load()
    x = _np(x_row_bf16, np.uint16).reshape(-1)
    y = np.empty((cfg.hidden,), np.float64)
    c = _cfg(cfg, act_quant)
    lib.orc_shared_row(ctypes.byref(c), ctypes.byref(weights.struct), _ptr(x), _ptr(y))
    return y


def forward_tokens(cfg, weights: Weights, x_bf16, ids, w, tokens=None, residual_bf16=None,
                   act_quant=True) -> np.ndarray:
    """Layer output (fp64) for the listed tokens, given the routing ids/w of all tokens."""
    lib = _load()
    x = _np(x_bf16, np.uint16)
    T = x.shape[0]
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(
        np.asarray(tokens, dtype=np.int32))
    r = _np(residual_bf16, np.uint16)
    out = np.empty((len(tokens), cfg.hidden), np.float64)
    c = _cfg(cfg, act_quant)
    lib.orc_forward_tokens(ctypes.byref(c), ctypes.byref(weights.struct), _ptr(x), _ptr(ids), _ptr(w),
                           _ptr(r), _ptr(tokens), len(tokens), _ptr(out))
    return out


def forward_tokens_mx(cfg, weights: WeightsMX, x_bf16, ids, w, tokens=None, residual_bf16=None,
                      act_quant=True) -> np.ndarray:
    """MXFP8 layer output (fp64) for the listed tokens, given the routing of all tokens."""
    lib = _load()
    x = _np(x_bf16, np.uint16)
    T = x.shape[0]
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(
        np.asarray(tokens, dtype=np.int32))
    r = _np(residual_bf16, np.uint16)
    out = np.empty((len(tokens), cfg.hidden), np.float64)
    c = _cfg(cfg, act_quant)
    lib.orc_forward_tokens_mx(ctypes.byref(c), ctypes.byref(weights.struct), _ptr(x), _ptr(ids), _ptr(w),
                              _ptr(r), _ptr(tokens), len(tokens), _ptr(out))
    return out


def forward_rmsnorm(cfg, weights_dict, h_bf16, gamma_bf16, eps: float, tokens=None, act_quant=True):
    """Stage M in front of the layer, the residual after it: out = h + layer(RMSNorm(h))."""
    x = rmsnorm(h_bf16, gamma_bf16, eps)
    return forward(cfg, weights_dict, x, tokens=tokens, residual_bf16=_np(h_bf16, np.uint16),
                   act_quant=act_quant)


def forward(cfg, weights_dict, x_bf16, bias=None, w_router=None, tokens=None, residual_bf16=None,
            act_quant=True):
    """Whole layer: route every token, then the output of the listed tokens."""
    W = Weights(weights_dict)
    ids, w, p, m = route(cfg, x_bf16, weights_dict["w_router"] if w_router is None else w_router,
                         weights_dict.get("router_bias") if bias is None else bias)
    out = forward_tokens(cfg, W, x_bf16, ids, w, tokens, residual_bf16, act_quant)
    return out, ids, w, m


def _bf16_to_f64(x) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values; float arrays pass through as float64."""
    a = _np(x, np.uint16) if (hasattr(x, "dtype") and str(x.dtype) in ("torch.bfloat16", "uint16")) else None
    if a is None:
        return np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def forward_fixed_ids(cfg, weights: Weights, x, ids, w_router, bias=None, act_quant=True) -> np.ndarray:
    """Layer output (fp64, [T, H]) with the expert choice `ids` fixed and the routing
    weights recomputed from x: the function the backward differentiates. x is fp64
    [T, H] (or bf16 bit patterns), w_router / bias fp64 copies (any float array)."""
    lib = _load()
    xd = _bf16_to_f64(x)
    T = xd.shape[0]
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    wr = np.ascontiguousarray(np.asarray(w_router, dtype=np.float64))
    b = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float64))
    out = np.empty((T, cfg.hidden), np.float64)
    c = _cfg(cfg, act_quant)
    lib.orc_forward_fixed_ids_d(ctypes.byref(c), ctypes.byref(weights.struct), _ptr(wr), _ptr(b), _ptr(xd), T,
                                _ptr(ids), _ptr(out))
    return out


def backward(cfg, weights: Weights, x, ids, w, dout, w_router, bias=None, act_quant=True, dx_only=False) -> dict:
    """Gradients of sum(dout * out) for the layer with the expert choice `ids` and the
    routing weights `w` the forward applied ([T, k]). Returns fp64 arrays: dx [T,H],
    dw_gate, dw_up [E,I,H], dw_down [E,H,I], dws_gate, dws_up [Is,H], dws_down [H,Is]
    (zero-size when there are no shared experts), dw_router [E,H], dbias [E].
    dx_only: only dx (None for the rest), for a sample of tokens at large sizes."""
    lib = _load()
    xd = _bf16_to_f64(x)
    T, H = xd.shape
    E, I, k = cfg.n_routed, cfg.moe_inter, cfg.top_k
    Is = cfg.n_shared * I
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
    do = np.ascontiguousarray(np.asarray(dout, dtype=np.float64))
    wr = np.ascontiguousarray(np.asarray(w_router, dtype=np.float64))
    b = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float64))
    if dx_only:  # the listed tokens' dx only (exact for any subset of tokens)
        g = {"dx": np.empty((T, H)), "dw_gate": None, "dw_up": None, "dw_down": None, "dws_gate": None,
             "dws_up": None, "dws_down": None, "dw_router": None, "dbias": None}
    else:
        g = {"dx": np.empty((T, H)), "dw_gate": np.empty((E, I, H)), "dw_up": np.empty((E, I, H)),
             "dw_down": np.empty((E, H, I)), "dws_gate": np.zeros((Is, H)), "dws_up": np.zeros((Is, H)),
             "dws_down": np.zeros((H, Is)), "dw_router": np.empty((E, H)), "dbias": np.empty(E)}
    c = _cfg(cfg, act_quant)
    lib.orc_backward_d(ctypes.byref(c), ctypes.byref(weights.struct), _ptr(wr), _ptr(b), _ptr(xd), T, _ptr(ids),
                       _ptr(w), _ptr(do), _ptr(g["dx"]), _ptr(g["dw_gate"]), _ptr(g["dw_up"]), _ptr(g["dw_down"]),
                       _ptr(g["dws_gate"]), _ptr(g["dws_up"]), _ptr(g["dws_down"]), _ptr(g["dw_router"]),
                       _ptr(g["dbias"]))
    return g
