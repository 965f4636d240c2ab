"""Stage M (RMSNorm x gamma in front of the router) through the C ABI, against the oracle.

Stage M of the DSV2-236B-MegaKernel stage flowchart (MoE subgraph), the hidden
state normalised and scaled by gamma before the router, then the layer N..R with the residual h: out = h + layer(RMSNorm(h)).

Bars: moe_rmsnorm's bf16 values equal the oracle's, except where the oracle's exact
value lies so close to a rounding midpoint (1e-5 relative) that fp32 arithmetic may
round it the other way, and then by one bf16 step; routing ids bit-exact on
unflagged tokens; layer outputs within max|err| <= 2e-2 * max|ref| + 1e-3; the fused
entry points give bit-identical results to moe_rmsnorm followed by the unfused calls.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import MoEConfig, WORKLOADS, make_router, make_tokens, make_weights

from _helpers import assert_out_close, effective_routing, host_weights

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_gemv_gb300 import build
    build.build()
    oracle.build()
    B.lib()


def _gamma(H, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (1.0 + 0.25 * torch.randn(H, generator=g, device="cuda")).to(torch.bfloat16)


def _u16(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _near_midpoint(exact, rel=1e-5):
    a = np.abs(exact)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.exp2(np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7)
        d = np.abs(a / q - np.floor(a / q) - 0.5) * q / np.where(a > 0, a, 1.0)
    return (a > 0) & (d < rel)


def _raw_hidden(cfg, T, seed, scale=3.0):
    return (make_tokens(cfg, T, seed, "cuda", name="h").float() * scale).to(torch.bfloat16)


def _inputs(cfg, T, seed, rows=None):
    """Seeded hidden rows and gamma, with gamma adjusted so that, on the listed rows (all
    by default), every normalised value (per the oracle) lies at least 1e-5 (relative)
    from a bf16 rounding midpoint, beyond the error of fp32 arithmetic: stage M then has
    one answer there, and the layer after it can be held to the ordinary bars on those
    tokens (every token's routing and output depend on its own row only). A gamma entry
    whose column holds a value too close to a midpoint is moved one bf16 step up (that
    leaves every 1/rms unchanged), and the check repeats."""
    h = _raw_hidden(cfg, T, seed)
    gam = _gamma(cfg.hidden, seed)
    rows = np.arange(T) if rows is None else np.asarray(rows)
    hb, g = _u16(h)[rows], _u16(gam)
    for _ in range(200):
        _, ex = oracle.rmsnorm(hb, g, EPS, return_exact=True)
        cols = _near_midpoint(ex).any(axis=0)
        if not cols.any():
            return h, torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).cuda()
        g = np.where(cols, g + 1, g).astype(np.uint16)
    raise AssertionError("could not move the inputs away from rounding midpoints")


def _rows(T, n, seed):
    if n is None or n >= T:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    return np.sort(np.concatenate([[0, T - 1], rng.choice(np.arange(1, T - 1), n - 2, replace=False)])).astype(
        np.int32)


@pytest.mark.parametrize("T,H", [(1, 5120), (5, 512), (64, 7168), (300, 1024)])
def test_rmsnorm_matches_oracle(T, H):
    cfg = MoEConfig(H, 128, 8, 1, 1, 1, 1.0, 0)
    h = _raw_hidden(cfg, T, 90 + T)
    h[0, :] = 0  # eps keeps an all-zero row finite
    gam = _gamma(H, T)
    x = torch.empty_like(h)
    B.moe_rmsnorm(h, gam, EPS, x)
    torch.cuda.synchronize()
    ref, exact = oracle.rmsnorm(_u16(h), _u16(gam), EPS, return_exact=True)
    got = _u16(x)
    diff = got != ref
    assert not (diff & ~_near_midpoint(exact)).any(), f"{int(diff.sum())} values differ away from a midpoint"
    step = np.abs(got.view(np.int16).astype(np.int32) - ref.view(np.int16).astype(np.int32))
    assert np.all(step[diff] == 1)
    assert not (got[0] & 0x7FFF).any()  # +-0 (the sign follows gamma's)


# Checked rows: all of them up to T = 64, a sample of 64 tokens at T = 4096.
@pytest.mark.parametrize("name,n", [("tiny_t8", None), ("dsv2_decode_t1", None), ("dsv2_decode_t64", None),
                                    ("prefill_t4096", 64)])
def test_route_rmsnorm(name, n):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    wr, bias = make_router(cfg, wl.seed, "cuda", zipf=wl.zipf_bias)
    rows = _rows(wl.T, n, wl.seed)
    h, gam = _inputs(cfg, wl.T, wl.seed, rows)
    ids = torch.empty((wl.T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, cfg.top_k), dtype=torch.float32, device="cuda")
    ws = B.alloc_workspace(cfg, wl.T)
    B.moe_route_rmsnorm(cfg, h, gam, EPS, wr, bias, ids, w, ws)
    x = torch.empty_like(h)
    B.moe_rmsnorm(h, gam, EPS, x)
    ids2, w2 = torch.empty_like(ids), torch.empty_like(w)
    B.moe_route(cfg, x, wr, bias, ids2, w2, B.alloc_workspace(cfg, wl.T))
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws) == 0
    assert torch.equal(ids, ids2) and torch.equal(w, w2), "fused stage M differs from moe_rmsnorm"
    xn = oracle.rmsnorm(_u16(h)[rows], _u16(gam), EPS)
    assert np.array_equal(_u16(x)[rows], xn)
    ids_o, w_o, p_o, margin = oracle.route(cfg, xn, wr.cpu(), None if bias is None else bias.cpu())
    _, w_eff, _ = effective_routing(cfg, ids.cpu().numpy()[rows], ids_o, p_o, margin)
    np.testing.assert_allclose(w.cpu().numpy()[rows], w_eff, rtol=2e-5, atol=1e-7)


def _check_forward(cfg, W, h, gam, tokens):
    T = h.shape[0]
    ws = B.alloc_workspace(cfg, T)
    out = torch.empty_like(h)
    ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    B.moe_forward_rmsnorm(cfg, h, gam, EPS, W, out, ids, ws)
    # the same layer unfused: stage M on its own, then moe_forward with residual h
    x = torch.empty_like(h)
    B.moe_rmsnorm(h, gam, EPS, x)
    out2 = torch.empty_like(h)
    ids2 = torch.empty_like(ids)
    B.moe_forward(cfg, x, W, out2, residual=h, topk_ids_out=ids2, ws=B.alloc_workspace(cfg, T))
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws) == 0
    assert torch.equal(ids, ids2) and torch.equal(out, out2), "fused stage M differs from moe_rmsnorm"
    Wc = host_weights(W)
    hb = _u16(h)[tokens]
    xn = oracle.rmsnorm(hb, _u16(gam), EPS)
    assert np.array_equal(_u16(x)[tokens], xn)  # the inputs leave stage M one answer there
    ids_o, w_o, p_o, margin = oracle.route(cfg, xn, Wc["w_router"], Wc["router_bias"])
    ids_eff, w_eff, _ = effective_routing(cfg, ids.cpu().numpy()[tokens], ids_o, p_o, margin)
    ref = oracle.forward_tokens(cfg, oracle.Weights(Wc), xn, ids_eff, w_eff, residual_bf16=hb)
    assert_out_close(out[torch.from_numpy(tokens).long().cuda()], ref, f"{cfg} T={T}")


@pytest.mark.parametrize("name,n", [("tiny_t8", None), ("dsv2_decode_t1", None), ("dsv2_decode_t64", 6),
                                    ("prefill_t4096", 6)])
def test_forward_rmsnorm_workloads(name, n):
    wl = WORKLOADS[name]
    W = make_weights(wl.cfg, wl.seed, "cuda", zipf=wl.zipf_bias)
    rows = _rows(wl.T, n, wl.seed)
    h, gam = _inputs(wl.cfg, wl.T, wl.seed, rows)
    _check_forward(wl.cfg, W, h, gam, rows)
    del W
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 33, 65, 257])
def test_forward_rmsnorm_ragged(T):
    cfg = MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 2)
    W = make_weights(cfg, 95, "cuda")
    h, gam = _inputs(cfg, T, 96 + T)
    _check_forward(cfg, W, h, gam, np.arange(T, dtype=np.int32))
