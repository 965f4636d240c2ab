"""moe_route_noalloc: the router + top-k for callers that cannot allocate device
memory (a framework that owns the whole memory pool and forbids cudaMalloc while
serving, or a plugin inside one). It must give what moe_route gives, on two calls
in a row: the second call reuses the library's one scratch array, so stale state
from the first call would show up here.

Collected last on purpose (file name), so a stop-at-first-failure run has already
run every other test when this one runs."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, MoEConfig, make_router, make_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_gemv_gb300 import build
    build.build()
    B.lib()


def _route_both(cfg, x, wr, bias):
    T = x.shape[0]
    ids_a = torch.full((T, cfg.top_k), -1, dtype=torch.int32, device="cuda")
    w_a = torch.zeros((T, cfg.top_k), dtype=torch.float32, device="cuda")
    ids_b = torch.full_like(ids_a, -2)
    w_b = torch.full_like(w_a, -1.0)
    ws = B.alloc_workspace(cfg, T)
    B.moe_route(cfg, x, wr, bias, ids_a, w_a, ws)
    B.moe_route_noalloc(cfg, x, wr, bias, ids_b, w_b)
    torch.cuda.synchronize()
    return ids_a.cpu().numpy(), w_a.cpu().numpy(), ids_b.cpu().numpy(), w_b.cpu().numpy()


@pytest.mark.parametrize("name,T", [("dsv2_decode_t64", 64), ("dsv2_decode_t1", 1), ("tiny_t8", 8)])
def test_noalloc_route_matches_route_on_two_calls_in_a_row(name, T):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    wr, bias = make_router(cfg, wl.seed, "cuda")
    for call in range(2):  # different tokens on each call
        x = make_tokens(cfg, T, wl.seed, "cuda", name=f"x_noalloc{call}")
        ids_a, w_a, ids_b, w_b = _route_both(cfg, x, wr, bias)
        assert np.array_equal(ids_a, ids_b), f"call {call}"
        np.testing.assert_allclose(w_b, w_a, rtol=2e-5, atol=1e-7)


def test_noalloc_route_with_bias_and_a_smaller_call_after_a_larger_one():
    cfg = MoEConfig(512, 256, 16, 4, 2, 4, 1.5, 0)
    wr, _ = make_router(cfg, 5, "cuda")
    bias = torch.linspace(-1.0, 1.0, 16, device="cuda")
    for T in (40, 3):
        x = make_tokens(cfg, T, 6 + T, "cuda")
        ids_a, w_a, ids_b, w_b = _route_both(cfg, x, wr, bias)
        assert np.array_equal(ids_a, ids_b)
        np.testing.assert_allclose(w_b, w_a, rtol=2e-5, atol=1e-7)


def test_noalloc_route_rejects_sizes_beyond_its_scratch():
    cfg = WORKLOADS["prefill_t4096"].cfg  # hidden 7168 fits; T = 65 does not
    wr, _ = make_router(cfg, 3, "cuda")
    x = make_tokens(cfg, 65, 3, "cuda")
    ids = torch.empty((65, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((65, cfg.top_k), dtype=torch.float32, device="cuda")
    with pytest.raises(B.MoeError) as e:
        B.moe_route_noalloc(cfg, x, wr, None, ids, w)
    assert e.value.status == -2
