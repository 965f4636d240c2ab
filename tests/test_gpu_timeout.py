"""Failure detection on the GPU, in the permitted form: a bounded device-side wait is made
to run out by a flag that nothing sets (moe_debug_set makes the decode gate/up kernel
issue no copies; its consumers' waits give up after about one second). The call must come
back with the timeout recorded in the workspace (moe_read_device_status ->
MOE_ERR_DEVICE_TIMEOUT) instead of hanging, with nothing left in flight, and the next
normal call on the same workspace must give the oracle's result again."""
import time

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, make_tokens, make_weights

from _helpers import assert_out_close, effective_routing, host_weights

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = -5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_gemv_gb300 import build
    build.build()
    oracle.build()
    B.lib()


@pytest.mark.parametrize("name", ["tiny_t8", "dsv2_decode_t1"])
def test_injected_wait_timeout_is_reported_and_the_workspace_recovers(name):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    W = make_weights(cfg, wl.seed, "cuda")
    x = make_tokens(cfg, wl.T, wl.seed, "cuda")
    ws = B.alloc_workspace(cfg, wl.T)
    ref = torch.empty_like(x)
    B.moe_forward(cfg, x, W, ref, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws) == 0

    B.moe_debug_set(ws, inject=B.INJECT_SKIP_GATEUP_LOADS)
    out = torch.empty_like(x)
    t0 = time.perf_counter()
    B.moe_forward(cfg, x, W, out, ws=ws)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert B.moe_read_device_status(ws) == MOE_ERR_DEVICE_TIMEOUT
    assert B.moe_read_device_status(ws) == 0  # the read clears it
    assert elapsed < 10.0, f"the timed-out call took {elapsed:.2f} s"  # the waits give up after ~1 s

    B.moe_debug_set(ws, inject=0)
    again = torch.empty_like(x)
    ids = torch.empty((wl.T, cfg.top_k), dtype=torch.int32, device="cuda")
    B.moe_forward(cfg, x, W, again, topk_ids_out=ids, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws) == 0
    assert torch.equal(again, ref)
    Wc = host_weights(W)
    ids_o, _, p_o, margin = oracle.route(cfg, x.cpu(), Wc["w_router"], Wc["router_bias"])
    ids_eff, w_eff, _ = effective_routing(cfg, ids.cpu().numpy(), ids_o, p_o, margin)
    tokens = np.arange(wl.T, dtype=np.int32)
    assert_out_close(again, oracle.forward_tokens(cfg, oracle.Weights(Wc), x.cpu(), ids_eff, w_eff, tokens), name)
