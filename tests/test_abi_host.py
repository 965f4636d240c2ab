"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
entry point include/moe.h declares, sizes its workspace, and rejects bad arguments
before launching anything."""
import ctypes
import dataclasses

import pytest

from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300 import build
from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, MoEConfig


@pytest.fixture(scope="module")
def L():
    build.build()
    return B.lib()


def test_exports_every_declared_symbol(L):
    names = B.declared_symbols()
    assert {"moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(0, -6, -1):
        assert B.status_string(code) not in ("", "unknown status")
    assert B.status_string(7) == "unknown status"


def test_workspace_size_grows_with_tokens_and_rejects_bad_configs(L):
    cfg = WORKLOADS["dsv2_decode_t1"].cfg
    sizes = [B.moe_workspace_size(cfg, t) for t in (0, 1, 64, 65, 4096)]
    assert all(s > 0 for s in sizes)
    assert sizes == sorted(sizes)
    bad = [dataclasses.replace(cfg, hidden=5000), dataclasses.replace(cfg, moe_inter=1500),
           dataclasses.replace(cfg, n_group=7), dataclasses.replace(cfg, topk_group=9),
           dataclasses.replace(cfg, top_k=17), dataclasses.replace(cfg, n_routed=300, n_group=10),
           dataclasses.replace(cfg, top_k=61), dataclasses.replace(cfg, n_shared=-1),
           dataclasses.replace(cfg, routed_scaling_factor=float("inf"))]
    for c in bad:
        assert B.moe_workspace_size(c, 1) == 0, c
    assert B.moe_workspace_size(cfg, -1) == 0


FAKE = 0x10000  # an aligned address that is never dereferenced: every call below fails its checks first


def _call_forward(cfg, T, x=FAKE, out=FAKE, ws=FAKE, ws_bytes=None, wfields=None):
    c = B.config_struct(cfg)
    W = B.moe_weights_t(*([FAKE] * 13 + [None]))
    for k, v in (wfields or {}).items():
        setattr(W, k, v)
    ws_bytes = B.moe_workspace_size(cfg, max(T, 0)) if ws_bytes is None else ws_bytes
    return B.lib().moe_forward(ctypes.byref(c), x, T, ctypes.byref(W), None, out, None, ws, ws_bytes, None)


def test_forward_argument_checks(L):
    cfg = WORKLOADS["tiny_t8"].cfg
    assert _call_forward(cfg, 0) == 0                                   # T = 0: no-op
    assert _call_forward(cfg, -1) == -1                                 # negative T
    assert _call_forward(cfg, 4, x=None) == -1                          # NULL input
    assert _call_forward(cfg, 4, out=FAKE + 4) == -1                    # misaligned output
    assert _call_forward(cfg, 4, ws=None) == -3                         # no workspace
    assert _call_forward(cfg, 4, ws_bytes=1024) == -3                   # workspace too small
    assert _call_forward(cfg, 4, wfields={"w_gate": None}) == -1        # missing weight
    assert _call_forward(cfg, 4, wfields={"ws_down": None}) == -1       # shared weight missing, n_shared = 1
    assert _call_forward(dataclasses.replace(cfg, hidden=500), 4) == -2  # H not a multiple of 128
    assert _call_forward(dataclasses.replace(cfg, top_k=9), 4) == -2     # k > Gk * E / G


def test_stage_argument_checks(L):
    cfg = WORKLOADS["tiny_t8"].cfg
    c = B.config_struct(cfg)
    lib = B.lib()
    ws_bytes = B.moe_workspace_size(cfg, 8)
    assert lib.moe_route(ctypes.byref(c), None, 8, FAKE, None, FAKE, FAKE, FAKE, ws_bytes, None) == -1
    assert lib.moe_route(ctypes.byref(c), FAKE, 8, FAKE, FAKE + 2, FAKE, FAKE, FAKE, ws_bytes, None) == -1
    assert lib.moe_permute(ctypes.byref(c), FAKE, 8, FAKE, FAKE, None, FAKE, ws_bytes, None) == -1
    assert lib.moe_permute(ctypes.byref(c), FAKE, 8, FAKE, FAKE, FAKE, FAKE, 16, None) == -3
    assert lib.moe_combine(ctypes.byref(c), FAKE, None, None, None, 8, FAKE, None) == -1
    assert lib.moe_combine(None, FAKE, FAKE, None, None, 8, FAKE, None) == -1
    assert lib.moe_quant_act(FAKE, 3, 100, FAKE, FAKE, None) == -2
    assert lib.moe_quant_act(FAKE, -3, 128, FAKE, FAKE, None) == -1
    assert lib.moe_quant_act(FAKE, 0, 128, FAKE, FAKE, None) == 0
    W = B.moe_weights_t(*([FAKE] * 14))
    assert lib.moe_expert_ffn(ctypes.byref(c), FAKE, 8, ctypes.byref(W), FAKE, FAKE, FAKE, FAKE, None, FAKE,
                              B.moe_workspace_size(cfg, 8), None) == -1  # y_shared required with n_shared > 0
    assert lib.moe_workspace_init(None, 256, None) == -3
    assert lib.moe_workspace_init(FAKE, 100, None) == -3


def test_workspace_covers_the_largest_workload(L):
    wl = WORKLOADS["prefill_t4096"]
    n = B.moe_workspace_size(wl.cfg, wl.T)
    c = wl.cfg
    # at least the permuted FP8 intermediate [T*k, I] and the bf16 expert outputs [T*k, H]
    assert n >= wl.T * c.top_k * (c.moe_inter + 2 * c.hidden)
    assert n < 4 * 1024 ** 3  # fp32 partial sums of the weight-streaming path dominate


def test_backward_workspace_and_argument_checks(L):
    c = B.config_struct(MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 1))
    n = L.moe_backward_workspace_size(ctypes.byref(c), 64)
    assert n > L.moe_backward_workspace_size(ctypes.byref(c), 8) > 0
    # unsupported: hidden not a multiple of 256, n_routed not a multiple of 16
    assert L.moe_backward_workspace_size(ctypes.byref(B.config_struct(MoEConfig(384, 256, 16, 4, 2, 4, 1.0, 1))), 8) == 0
    assert L.moe_backward_workspace_size(ctypes.byref(B.config_struct(MoEConfig(512, 256, 8, 4, 2, 4, 1.0, 1))), 8) == 0
    w = B.moe_weights_t()
    # no weights / no gradient outputs: rejected before anything is launched
    assert L.moe_backward(ctypes.byref(c), None, 8, None, None, None, None, None, None, None, None, None, None,
                          None, None, None, None, 0, None) == -1
    assert L.moe_backward(ctypes.byref(c), None, 8, ctypes.byref(w), None, None, None, None, None, None, None,
                          None, None, None, None, None, None, 0, None) == -1


def test_debug_set_checks_its_arguments_before_any_device_work():
    from mixture_experts_layer_gemv_gb300 import binding as B
    lib = B.lib()
    assert lib.moe_debug_set(None, 4096, 0, None) == -3                 # MOE_ERR_WORKSPACE
    assert lib.moe_debug_set(ctypes.c_void_p(4096), 16, 0, None) == -3  # below the control region
    assert lib.moe_debug_set(ctypes.c_void_p(4096), 4096, 2, None) == -1  # unknown inject bit
