"""The MXFP8 variant through the C ABI against the oracle: E4M3 codes with one UE8M0
scale per row and 32 consecutive K for weights and activations; the grouped GEMM (T > 64)
applies the scales inside the tensor core (tcgen05.mma kind::mxf8f6f4), the
weight-streaming kernels (T <= 64) per 32-wide MMA partial.

Bars: activation codes and scale bytes bit-exact; expert ids bit-exact on unflagged
tokens (routing is moe_route's); outputs within max|err| <= 2e-2 * max|ref| + 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import MoEConfig, WORKLOADS, make_tokens, make_weights_mx

from _helpers import assert_out_close, effective_routing, host_weights

pytestmark = pytest.mark.gpu

MX_CFG = MoEConfig(512, 512, 16, 4, 2, 4, 1.0, 1)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_gemv_gb300 import build
    build.build()
    oracle.build()
    B.lib()


@pytest.mark.parametrize("T,H", [(1, 5120), (8, 512), (37, 7168), (300, 1024)])
def test_quant_act_mx_bit_exact(T, H):
    g = torch.Generator(device="cuda").manual_seed(T * 5 + H)
    x = (torch.randn((T, H), generator=g, device="cuda") *
         torch.exp2(torch.randint(-12, 12, (T, H // 32), generator=g, device="cuda").float()).repeat_interleave(
             32, dim=1)).to(torch.bfloat16)
    x[0, :32] = 0
    x[0, 64:96] = 448.0  # on a scale boundary
    xq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    B.moe_quant_act_mx(x, xq, xs)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_rows_mx(x.float().cpu().numpy().astype(np.float64))
    assert np.array_equal(xs.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), q_ref)


def _check(cfg, W, x, tokens=None, residual=None):
    out, ids = B.forward_mx(cfg, x, W, residual=residual, return_ids=True)
    torch.cuda.synchronize()
    Wc = host_weights(W)
    ids_o, w_o, p_o, margin = oracle.route(cfg, x.cpu(), Wc["w_router"], Wc["router_bias"])
    ids_eff, w_eff, _ = effective_routing(cfg, ids.cpu().numpy(), ids_o, p_o, margin)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else tokens
    ref = oracle.forward_tokens_mx(cfg, oracle.WeightsMX(Wc), x.cpu(), ids_eff, w_eff, tokens,
                                   residual_bf16=None if residual is None else residual.cpu())
    assert_out_close(out[torch.from_numpy(tokens).long().cuda()], ref, f"{cfg} T={T}")
    return out


@pytest.mark.parametrize("T", [1, 37, 129, 300])
def test_forward_mx_ragged(T):
    W = make_weights_mx(MX_CFG, 110, "cuda")
    x = make_tokens(MX_CFG, T, 111 + T, "cuda")
    res = make_tokens(MX_CFG, T, 112, "cuda", name="residual")
    _check(MX_CFG, W, x, residual=res)


@pytest.mark.parametrize("T", [7, 200])  # weight-streaming path, grouped GEMM
def test_forward_mx_scrambled_scales(T):
    """Scale bytes that differ strongly between the 32-blocks of every row (weights and
    activations), so a scale applied to the wrong K step or row shows at once."""
    W = make_weights_mx(MX_CFG, 120, "cuda")
    g = torch.Generator(device="cuda").manual_seed(121)
    for k in ("s_gate", "s_up", "s_down", "ss_gate", "ss_up", "ss_down"):
        W[k] = (W[k].int() + torch.randint(-3, 4, W[k].shape, generator=g, device="cuda")).to(torch.uint8)
    x = make_tokens(MX_CFG, T, 122, "cuda").float()
    x = (x * torch.exp2(torch.randint(-4, 5, (T, MX_CFG.hidden // 32), generator=g, device="cuda").float())
         .repeat_interleave(32, dim=1)).to(torch.bfloat16)
    _check(MX_CFG, W, x)


@pytest.mark.parametrize("name,n", [("dsv2_decode_t1", None), ("dsv2_decode_t64", 8), ("prefill_t4096", 8),
                                    ("dsv2_zipf_t2048", 8)])
def test_forward_mx_workloads(name, n):
    wl = WORKLOADS[name]
    W = make_weights_mx(wl.cfg, wl.seed, "cuda", zipf=wl.zipf_bias)
    x = make_tokens(wl.cfg, wl.T, wl.seed, "cuda")
    tokens = None
    if n is not None:
        rng = np.random.default_rng(wl.seed)
        tokens = np.sort(np.concatenate([[0, wl.T - 1], rng.choice(np.arange(1, wl.T - 1), n - 2, replace=False)]))
        tokens = tokens.astype(np.int32)
    _check(wl.cfg, W, x, tokens)
    del W
    torch.cuda.empty_cache()


def test_mx_shape_rules():
    assert B.moe_workspace_size_mx(MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 1), 8) == 0  # moe_inter % 512
    assert B.moe_workspace_size_mx(MX_CFG, 8) > 0
