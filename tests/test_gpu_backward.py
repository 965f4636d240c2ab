"""Parity of the layer backward (moe_backward) with the oracle's fp64 backward.

The backward differentiates sum(dout * out) with the forward's expert choice fixed
(Mixture-of-Kittens, Table 1 "Backward"); both sides get the routing the GPU forward
chose (moe_route) and the same seeded dout. Every gradient tensor must satisfy
max|err| <= 2e-2 * max|ref| + 1e-3, the layer output's bound: the GPU contracts in
bf16 with fp32 accumulation (one bf16 rounding of each dequantised weight and of the
SwiGLU gradients, ~2^-9 relative), against fp64. At the prefill shape the oracle
checks dx of a sample of tokens (exact for any subset, since dx_t depends on token t
alone) and the router's gradient property (every token's dlogit sums to zero).
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, MoEConfig, make_tokens, make_weights

pytestmark = pytest.mark.gpu


def _route(cfg, x, W):
    T = x.shape[0]
    ws = B.alloc_workspace(cfg, T)
    ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.top_k), dtype=torch.float32, device="cuda")
    B.moe_route(cfg, x, W["w_router"], W["router_bias"], ids, w, ws)
    return ids, w


def _dout(cfg, T, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn((T, cfg.hidden), generator=g).to(torch.bfloat16).cuda()


def _f64(t):
    return None if t is None else t.detach().cpu().double().numpy()


def _close(name, got, ref):
    err = float(np.abs(got - ref).max())
    bound = 2e-2 * float(np.abs(ref).max()) + 1e-3
    assert err <= bound, (name, err, bound)


def _oracle(cfg, W, x, ids, w, dout, rows=None, dx_only=False):
    sel = slice(None) if rows is None else rows
    return oracle.backward(cfg, oracle.Weights(W), x[sel], ids.cpu().numpy()[sel], _f64(w)[sel], _f64(dout)[sel],
                           _f64(W["w_router"]), _f64(W["router_bias"]), dx_only=dx_only)


CASES = [
    ("tiny", MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 1), 8, 0, False),
    ("ragged tiles, two shared", MoEConfig(1024, 512, 32, 4, 2, 4, 2.5, 2), 300, 1, False),
    ("no shared experts", MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 0), 70, 2, False),
    ("router bias", MoEConfig(512, 256, 16, 4, 2, 4, 16.0, 1), 40, 3, True),
]


@pytest.mark.parametrize("name,cfg,T,seed,zipf", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(name, cfg, T, seed, zipf):
    W = make_weights(cfg, seed, "cuda", zipf=zipf)
    x = make_tokens(cfg, T, seed + 100, "cuda")
    ids, w = _route(cfg, x, W)
    dout = _dout(cfg, T, seed + 7)
    ws = B.alloc_workspace_backward(cfg, T)
    g = B.alloc_grads(cfg, T)
    B.moe_backward(cfg, x, W, ids, w, dout, g, ws)
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws) == 0
    ref = _oracle(cfg, W, x, ids, w, dout)
    for k, v in g.items():
        r = ref[k]
        if r is None or r.size == 0:
            continue
        _close(k, v.cpu().double().numpy(), r)


def test_backward_is_deterministic():
    cfg = MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 1)
    W = make_weights(cfg, 5, "cuda")
    x = make_tokens(cfg, 100, 6, "cuda")
    ids, w = _route(cfg, x, W)
    dout = _dout(cfg, 100, 7)
    a = B.backward(cfg, x, W, ids, w, dout)
    b = B.backward(cfg, x, W, ids, w, dout)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_zero_tokens_zero_weight_gradients():
    cfg = MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 1)
    W = make_weights(cfg, 5, "cuda")
    x = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    w = torch.empty((0, 4), dtype=torch.float32, device="cuda")
    g = B.alloc_grads(cfg, 0)
    for v in g.values():
        v.fill_(7.0)
    ws = B.alloc_workspace_backward(cfg, 1)
    B.moe_backward(cfg, x, W, ids, w, x, g, ws)
    torch.cuda.synchronize()
    for k, v in g.items():
        assert bool((v == 0).all()), k


def test_backward_prefill_shape_sampled_tokens():
    wl = WORKLOADS["prefill_t4096"]
    cfg, T = wl.cfg, wl.T
    W = make_weights(cfg, wl.seed, "cuda")
    x = make_tokens(cfg, T, 100, "cuda")
    ids, w = _route(cfg, x, W)
    dout = _dout(cfg, T, 11)
    g = B.backward(cfg, x, W, ids, w, dout)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 777, 2048, T - 2, T - 1])
    ref = _oracle(cfg, W, x, ids, w, dout, rows=rows, dx_only=True)
    _close("dx (sampled tokens)", g["dx"][rows].cpu().double().numpy(), ref["dx"])
    # every token's softmax gradient sums to zero, so dbias (their sum) does too
    db = g["dbias"].double()
    assert abs(float(db.sum())) <= 1e-3 * float(db.abs().sum()) + 1e-6
    for k, v in g.items():
        assert bool(torch.isfinite(v).all()), k


@pytest.mark.parametrize("name", ["dsv2_zipf_t2048", "dsv2_decode_t64"])
def test_backward_dsv2_shape_sampled_tokens(name):
    # E = 160 (two 128-row tiles of the router's weight gradient), I = 1536 (six 256-column
    # tiles), two shared experts; the load-imbalance workload adds the router bias
    wl = WORKLOADS[name]
    cfg, T = wl.cfg, wl.T
    W = make_weights(cfg, wl.seed, "cuda", zipf=wl.zipf_bias)
    x = make_tokens(cfg, T, 300, "cuda")
    ids, w = _route(cfg, x, W)
    dout = _dout(cfg, T, 13)
    g = B.backward(cfg, x, W, ids, w, dout)
    torch.cuda.synchronize()
    rows = np.unique(np.array([0, 5, T // 2, T - 1]))
    ref = _oracle(cfg, W, x, ids, w, dout, rows=rows, dx_only=True)
    _close("dx (sampled tokens)", g["dx"][rows].cpu().double().numpy(), ref["dx"])
    db = g["dbias"].double()
    assert abs(float(db.sum())) <= 1e-3 * float(db.abs().sum()) + 1e-6


def test_backward_invalid_expert_id_is_reported_not_faulted():
    cfg = MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 1)
    W = make_weights(cfg, 5, "cuda")
    x = make_tokens(cfg, 16, 6, "cuda")
    ids, w = _route(cfg, x, W)
    ids[3, 1] = 99  # >= n_routed
    dout = _dout(cfg, 16, 7)
    ws = B.alloc_workspace_backward(cfg, 16)
    g = B.alloc_grads(cfg, 16)
    B.moe_backward(cfg, x, W, ids, w, dout, g, ws)
    assert B.moe_read_device_status(ws) == -1  # MOE_ERR_INVALID_ARG
    assert B.moe_read_device_status(ws) == 0
