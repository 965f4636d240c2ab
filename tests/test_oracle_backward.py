"""Pins of the oracle's layer backward (dx, expert and router weight gradients).

The backward differentiates L = sum(dout * out) for the layer with the expert choice
held fixed (selection is piecewise constant) and the routing weights w = s * p_e
recomputed from x (Mixture-of-Kittens, Table 1 "Backward"; the formulas are the
reading taken here, not printed on the pages). It is pinned by central finite
differences of the oracle's own forward with fixed ids (a separate code path: a
mistake in a chain-rule term changes the analytic gradient but not the forward), by
linearity in dout, by the routing weights' scale s = 0 limit, and by the FP8
straight-through reading (the down-weight gradient of a single routed row is exactly
w * dout (x) ahat, with ahat the forward's quantised intermediate).
"""
import numpy as np
import pytest

from mixture_experts_layer_gemv_gb300.synth import MoEConfig, make_weights, make_tokens

CFG = MoEConfig(128, 128, 8, 2, 1, 2, 2.5, 1)  # H, I, E, G, Gk, k, s, S
T = 3


def _setup(orc, cfg=CFG, seed=11, act_quant=False):
    W = make_weights(cfg, seed)
    x = make_tokens(cfg, T, seed + 1)
    w_router = W["w_router"].double().numpy() * 10.0  # sharper routing: softmax terms matter
    xd = orc._bf16_to_f64(x)
    logits = xd @ w_router.T
    ids, w, _, _ = orc.topk(cfg, logits)
    rng = np.random.default_rng(seed + 2)
    dout = rng.standard_normal((T, cfg.hidden))
    return W, orc.Weights(W), xd, w_router, ids, w, dout


def _loss(orc, cfg, Wo, x, ids, w_router, dout, act_quant=False, bias=None):
    return float(np.sum(dout * orc.forward_fixed_ids(cfg, Wo, x, ids, w_router, bias, act_quant)))


def test_dx_matches_central_differences(orc):
    W, Wo, x, wr, ids, w, dout = _setup(orc)
    g = orc.backward(CFG, Wo, x, ids, w, dout, wr, act_quant=False)
    rng = np.random.default_rng(5)
    eps = 1e-5
    dirs = [rng.standard_normal(x.shape) for _ in range(4)]
    for t, h in ((0, 0), (1, 77), (2, 127)):  # single coordinates too
        v = np.zeros_like(x)
        v[t, h] = 1.0
        dirs.append(v)
    for v in dirs:
        fd = (_loss(orc, CFG, Wo, x + eps * v, ids, wr, dout) - _loss(orc, CFG, Wo, x - eps * v, ids, wr, dout)) / (
            2 * eps)
        an = float(np.sum(g["dx"] * v))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)


def test_router_gradients_match_central_differences(orc):
    W, Wo, x, wr, ids, w, dout = _setup(orc)
    bias = np.linspace(-0.1, 0.1, CFG.n_routed)
    g = orc.backward(CFG, Wo, x, ids, w, dout, wr, bias=bias, act_quant=False)
    rng = np.random.default_rng(6)
    eps = 1e-6
    for _ in range(3):
        v = rng.standard_normal(wr.shape)
        fd = (_loss(orc, CFG, Wo, x, ids, wr + eps * v, dout, bias=bias) -
              _loss(orc, CFG, Wo, x, ids, wr - eps * v, dout, bias=bias)) / (2 * eps)
        an = float(np.sum(g["dw_router"] * v))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)
    for e in (0, 3, 7):
        b1, b2 = bias.copy(), bias.copy()
        b1[e] += eps
        b2[e] -= eps
        fd = (_loss(orc, CFG, Wo, x, ids, wr, dout, bias=b1) - _loss(orc, CFG, Wo, x, ids, wr, dout, bias=b2)) / (
            2 * eps)
        assert abs(fd - g["dbias"][e]) <= 1e-6 * max(1.0, abs(fd)), (e, fd, g["dbias"][e])
    # the softmax gradient sums to zero over the experts of every token
    assert abs(g["dbias"].sum()) < 1e-9 * max(1.0, np.abs(g["dbias"]).max())


@pytest.mark.parametrize("name,scale_key,grad_key", [
    ("gate", "s_gate", "dw_gate"), ("up", "s_up", "dw_up"), ("down", "s_down", "dw_down"),
    ("shared gate", "ss_gate", "dws_gate"), ("shared up", "ss_up", "dws_up"), ("shared down", "ss_down", "dws_down")])
def test_weight_gradients_match_block_scale_differences(orc, name, scale_key, grad_key):
    # a block scale multiplies 128 x 128 dequantised weights: dL/ds = sum over the block
    # of dL/dW * code value; the scales are float32, so the step actually taken is used
    W, Wo, x, wr, ids, w, dout = _setup(orc)
    g = orc.backward(CFG, Wo, x, ids, w, dout, wr, act_quant=False)
    codes = W[{"s_gate": "w_gate", "s_up": "w_up", "s_down": "w_down", "ss_gate": "ws_gate", "ss_up": "ws_up",
               "ss_down": "ws_down"}[scale_key]].numpy()
    dec = orc.e4m3_decode(codes)
    for blk in ((0, 0, 0), (CFG.n_routed - 1, 0, 0)) if not name.startswith("shared") else ((None, 0, 0),):
        e, bo, bi = blk
        key_arr = Wo.arrays[scale_key]
        idx = (e, bo, bi) if e is not None else (bo, bi)
        s0 = np.float32(key_arr[idx])
        vals = []
        for sgn in (+1, -1):
            key_arr[idx] = np.float32(s0 * (1 + sgn * 1e-3))
            vals.append((float(key_arr[idx]), _loss(orc, CFG, Wo, x, ids, wr, dout)))
        key_arr[idx] = s0
        fd = (vals[0][1] - vals[1][1]) / (vals[0][0] - vals[1][0])
        gk = g[grad_key][e] if e is not None else g[grad_key]
        dk = dec[e] if e is not None else dec
        blkg = gk[128 * bo:128 * bo + 128, 128 * bi:128 * bi + 128]
        blkc = dk[128 * bo:128 * bo + 128, 128 * bi:128 * bi + 128]
        an = float(np.sum(blkg * blkc))
        assert abs(fd - an) <= 1e-5 * max(1e-3, abs(an)), (name, e, fd, an)


def test_backward_is_linear_in_dout(orc):
    W, Wo, x, wr, ids, w, dout = _setup(orc, act_quant=True)
    g1 = orc.backward(CFG, Wo, x, ids, w, dout, wr, act_quant=True)
    g2 = orc.backward(CFG, Wo, x, ids, w, 2.0 * dout, wr, act_quant=True)
    for k in g1:
        np.testing.assert_allclose(g2[k], 2.0 * g1[k], rtol=1e-12, atol=1e-300)


def test_zero_routed_scale_leaves_only_shared_gradients(orc):
    cfg = MoEConfig(128, 128, 8, 2, 1, 2, 0.0, 1)
    W, Wo, x, wr, ids, w, dout = _setup(orc, cfg=cfg)
    assert np.all(w == 0.0)
    g = orc.backward(cfg, Wo, x, ids, w, dout, wr, act_quant=True)
    for k in ("dw_gate", "dw_up", "dw_down", "dw_router", "dbias"):
        assert np.all(g[k] == 0.0), k
    assert np.any(g["dws_down"] != 0.0) and np.any(g["dx"] != 0.0)


def test_single_row_down_gradient_is_w_dout_times_quantised_intermediate(orc):
    # straight-through reading: the forward's FP8 intermediate ahat (not a) enters dWd
    cfg = MoEConfig(128, 128, 4, 1, 1, 1, 1.5, 0)
    W = make_weights(cfg, 3)
    Wo = orc.Weights(W)
    x = make_tokens(cfg, 1, 4)
    xd = orc._bf16_to_f64(x)
    wr = W["w_router"].double().numpy()
    ids, w, _, _ = orc.topk(cfg, xd @ wr.T)
    dout = np.random.default_rng(9).standard_normal((1, 128))
    g = orc.backward(cfg, Wo, x, ids, w, dout, wr, act_quant=True)
    e = int(ids[0, 0])
    _, a_hat = orc.expert_row(cfg, Wo, x[0], e, 1.0, act_quant=True)
    np.testing.assert_allclose(g["dw_down"][e], w[0, 0] * np.outer(dout[0], a_hat), rtol=1e-12, atol=1e-300)
    others = [i for i in range(cfg.n_routed) if i != e]
    assert np.all(g["dw_down"][others] == 0.0)
