"""Pins of the oracle's expert MLP, shared experts and whole-layer combine.

Stages P1/P2 (routed gate+up, SiLU(g) * u, down x w), Q1/Q2 (shared experts) and
R's local combine h = shared_out + routed of "DSV2-236B-MegaKernel" (README,
stage flowchart, MoE subgraph). Pinned by a hand-worked case
(tests/golden/swiglu_hand.txt), reductions to torch fp64 library routines on
dequantised weights, and the special cases the method reduces to (zero weight,
shared = routed expert with w = 1, two fused shared experts = two experts,
dense softmax mixture when every expert is selected).
"""
import math
import os

import numpy as np
import pytest
import torch

from mixture_experts_layer_gemv_gb300.synth import MoEConfig, make_weights, make_tokens

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "swiglu_hand.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        if line.startswith("act_quant_"):
            key, rest = line.split(None, 1)
            vals[key] = float(rest.split("=")[1])
    return vals


def _const_weights(cfg, gate_s, up_s, down_s):
    E, I, H = cfg.n_routed, cfg.moe_inter, cfg.hidden
    return {
        "w_gate": torch.full((E, I, H), 0x38, dtype=torch.uint8),
        "w_up": torch.full((E, I, H), 0x38, dtype=torch.uint8),
        "w_down": torch.full((E, H, I), 0x38, dtype=torch.uint8),
        "s_gate": torch.full((E, I // 128, H // 128), gate_s),
        "s_up": torch.full((E, I // 128, H // 128), up_s),
        "s_down": torch.full((E, H // 128, I // 128), down_s),
    }


def test_hand_swiglu_single_expert_single_token(orc):
    g = _golden()
    cfg = MoEConfig(128, 128, 1, 1, 1, 1, 1.0, 0)
    W = orc.Weights(_const_weights(cfg, 2.0 ** -7, 2.0 ** -6, 2.0 ** -7))
    x = torch.ones((1, 128), dtype=torch.bfloat16)
    y, a = orc.expert_row(cfg, W, x[0], 0, 0.75, act_quant=True)
    assert np.all(a == 1.5)
    assert np.all(y == g["act_quant_on"])
    y, a = orc.expert_row(cfg, W, x[0], 0, 0.75, act_quant=False)
    assert np.allclose(a, 2.0 / (1.0 + math.exp(-1.0)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(y, g["act_quant_off"], rtol=1e-13)  # 128-term fp64 sum


def _dequant(codes, scales):
    """Library dequantisation: torch float8 decode times the block scale broadcast."""
    v = codes.view(torch.float8_e4m3fn).to(torch.float64)
    s = scales.to(torch.float64)
    s = s.repeat_interleave(128, -2).repeat_interleave(128, -1)
    return v * s


def _bf16_f64(x):
    return x.to(torch.float64)


def _torch_expert(x, wg, sg, wu, su, wd, sd, w):
    g = _dequant(wg, sg) @ x
    u = _dequant(wu, su) @ x
    a = torch.nn.functional.silu(g) * u
    return w * (_dequant(wd, sd) @ a)


@pytest.fixture(scope="module")
def small_layer():
    cfg = MoEConfig(384, 256, 6, 2, 1, 2, 1.7, 2)
    W = make_weights(cfg, 11)
    x = make_tokens(cfg, 5, 11)
    return cfg, W, x


def test_expert_row_matches_torch_fp64_without_act_quant(orc, small_layer):
    cfg, W, x = small_layer
    OW = orc.Weights(W)
    for t, e, w in [(0, 0, 1.0), (3, 5, -0.25), (4, 2, 3.0)]:
        y, _ = orc.expert_row(cfg, OW, x[t], e, w, act_quant=False)
        ref = _torch_expert(_bf16_f64(x[t]), W["w_gate"][e], W["s_gate"][e], W["w_up"][e], W["s_up"][e],
                            W["w_down"][e], W["s_down"][e], w)
        np.testing.assert_allclose(y, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_act_quant_stays_within_fp8_error_of_unquantised(orc, small_layer):
    cfg, W, x = small_layer
    OW = orc.Weights(W)
    y_q, _ = orc.expert_row(cfg, OW, x[1], 3, 1.0, act_quant=True)
    y_f, _ = orc.expert_row(cfg, OW, x[1], 3, 1.0, act_quant=False)
    err = np.abs(y_q - y_f).max() / np.abs(y_f).max()
    assert 1e-4 < err < 0.1   # quantisation is applied, and only perturbs at the FP8 level


def test_zero_routing_weight_contributes_exactly_zero(orc, small_layer):
    cfg, W, x = small_layer
    y, _ = orc.expert_row(cfg, orc.Weights(W), x[2], 4, 0.0)
    assert np.all(y == 0.0)


def test_shared_expert_equals_routed_expert_with_weight_one(orc):
    cfg = MoEConfig(256, 128, 3, 1, 1, 1, 1.0, 1)
    W = make_weights(cfg, 12)
    for a, b in (("gate", "gate"), ("up", "up"), ("down", "down")):
        W[f"ws_{a}"] = W[f"w_{b}"][2].clone()
        W[f"ss_{a}"] = W[f"s_{b}"][2].clone()
    OW = orc.Weights(W)
    x = make_tokens(cfg, 2, 12)
    for aq in (True, False):
        ys = orc.shared_row(cfg, OW, x[1], act_quant=aq)
        yr, _ = orc.expert_row(cfg, OW, x[1], 2, 1.0, act_quant=aq)
        assert np.array_equal(ys, yr)


def test_two_fused_shared_experts_equal_two_separate_experts(orc):
    cfg = MoEConfig(256, 128, 2, 1, 1, 1, 1.0, 2)
    W = make_weights(cfg, 13)
    W["ws_gate"] = torch.cat([W["w_gate"][0], W["w_gate"][1]], 0)
    W["ss_gate"] = torch.cat([W["s_gate"][0], W["s_gate"][1]], 0)
    W["ws_up"] = torch.cat([W["w_up"][0], W["w_up"][1]], 0)
    W["ss_up"] = torch.cat([W["s_up"][0], W["s_up"][1]], 0)
    W["ws_down"] = torch.cat([W["w_down"][0], W["w_down"][1]], 1)
    W["ss_down"] = torch.cat([W["s_down"][0], W["s_down"][1]], 1)
    OW = orc.Weights(W)
    x = make_tokens(cfg, 1, 13)
    for aq in (True, False):
        ys = orc.shared_row(cfg, OW, x[0], act_quant=aq)
        y0, _ = orc.expert_row(cfg, OW, x[0], 0, 1.0, act_quant=aq)
        y1, _ = orc.expert_row(cfg, OW, x[0], 1, 1.0, act_quant=aq)
        np.testing.assert_allclose(ys, y0 + y1, rtol=1e-12, atol=1e-14)


def test_layer_with_every_expert_selected_is_dense_softmax_mixture(orc):
    # G = Gk = 1 and k = E: group-limited top-k keeps everything, so the layer is
    # sum_e softmax(logits)_e * s * expert_e(x) + shared(x)
    cfg = MoEConfig(256, 128, 4, 1, 1, 4, 2.0, 1)
    W = make_weights(cfg, 14)
    x = make_tokens(cfg, 3, 14)
    res = make_tokens(cfg, 3, 14, name="residual")
    out, ids, w, _ = orc.forward(cfg, W, x, residual_bf16=res, act_quant=False)
    xf = _bf16_f64(x)
    p = torch.softmax(xf @ W["w_router"].to(torch.float64).T, dim=1)
    for t in range(3):
        ref = _bf16_f64(res[t]).clone()
        for e in range(4):
            ref += _torch_expert(xf[t], W["w_gate"][e], W["s_gate"][e], W["w_up"][e], W["s_up"][e],
                                 W["w_down"][e], W["s_down"][e], float(p[t, e]) * 2.0)
        ref += _torch_expert(xf[t], W["ws_gate"], W["ss_gate"], W["ws_up"], W["ss_up"], W["ws_down"],
                             W["ss_down"], 1.0)
        np.testing.assert_allclose(out[t], ref.numpy(), rtol=1e-9, atol=1e-11)


def test_forward_sums_routed_rows_and_shared(orc, small_layer):
    cfg, W, x = small_layer
    out, ids, w, _ = orc.forward(cfg, W, x)
    OW = orc.Weights(W)
    for t in range(x.shape[0]):
        ref = orc.shared_row(cfg, OW, x[t])
        for j in range(cfg.top_k):
            y, _ = orc.expert_row(cfg, OW, x[t], ids[t, j], w[t, j])
            ref = ref + y
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-13)
