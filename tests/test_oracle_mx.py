"""Pins of the oracle's MXFP8 variant: E8M0 scale decode, per-32 quantisation, and the
MXFP8 expert MLP / layer.

The variant stores E4M3 codes with one UE8M0 (power-of-two) scale per 32 consecutive
values along K, for weights and activations (Mixture-of-Kittens Table 2, its MXFP8
routed-expert rows; the DeepSeek-V4.1 Flash lecture's conversion of block scales to the
MX layout and its MXFP8 quantisation of the experts' inputs). Pinned by torch's float8_e8m0fnu / float8_e4m3fn conversions (library
routines), the agreement with the per-128 quantiser when the four 32-blocks of a
128-block share their maximum, a hand-worked MLP (tests/golden/mx_swiglu_hand.txt) and
torch fp64 matmuls on dequantised weights.
"""
import math
import os

import numpy as np
import pytest
import torch

from mixture_experts_layer_gemv_gb300.synth import MoEConfig, make_tokens, make_weights_mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_swiglu_hand.txt")


def test_e8m0_decode_matches_torch(orc):
    b = np.arange(256, dtype=np.uint8)
    ours = orc.e8m0_decode(b)
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.from_numpy(b).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert np.array_equal(np.isnan(ours), np.isnan(ref))
        assert np.array_equal(ours[:255], ref[:255])
    assert np.isnan(ours[255]) and ours[127] == 1.0 and ours[0] == 2.0 ** -127 and ours[254] == 2.0 ** 127


def test_mx_quant_rule_and_codes(orc):
    rng = np.random.default_rng(5)
    v = rng.standard_normal((16, 256)) * np.exp(rng.standard_normal((16, 8)).repeat(32, axis=1) * 4)
    v[0, :32] = 0.0
    v[1, 32:64] = 448.0 * 2.0 ** -3  # exactly on a scale boundary
    q, s = orc.quant_rows_mx(v)
    k = s.astype(np.int64) - 127
    blocks = v.reshape(16, 8, 32)
    amax = np.abs(blocks).max(-1)
    sc = np.exp2(k.astype(np.float64))
    nz = amax > 0
    # the smallest power of two with amax <= 448 * scale
    assert np.all(amax[nz] <= 448 * sc[nz]) and np.all(amax[nz] > 448 * sc[nz] / 2)
    assert np.all(k[~nz] == 0) and not q[0, :32].any()
    assert k[1, 1] == -3
    # the codes are torch's RNE E4M3 conversion of v / scale
    ref = torch.from_numpy((blocks / sc[..., None]).reshape(16, 256)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(q, ref.numpy())


def test_mx_quant_agrees_with_per128_when_subblocks_share_the_max(orc):
    rng = np.random.default_rng(9)
    v = rng.uniform(-1, 1, (6, 512)) * np.exp2(rng.integers(-20, 20, (6, 4))).repeat(128, axis=1)
    b = v.reshape(6, 16, 32)
    m = np.abs(b).max(-1)
    big = m.reshape(6, 4, 4).max(-1).repeat(4, axis=1)  # every 32-block gets its 128-block's max
    b[np.arange(6)[:, None], np.arange(16)[None, :], np.abs(b).argmax(-1)] = big * np.sign(
        b[np.arange(6)[:, None], np.arange(16)[None, :], np.abs(b).argmax(-1)])
    v = b.reshape(6, 512)
    q_mx, s_mx = orc.quant_rows_mx(v)
    q, s = orc.quant_rows(v)
    assert np.array_equal(q_mx, q)
    assert np.array_equal(np.exp2(s_mx.astype(np.float64) - 127), np.repeat(s, 4, axis=1))


def _golden():
    vals = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_mx_mlp_hand_worked(orc):
    g = _golden()
    cfg = MoEConfig(64, 64, 1, 1, 1, 1, 1.0, 0)
    code = lambda shape: np.full(shape, 0x38, np.uint8)
    sd = np.empty((1, 64, 2), np.uint8)
    sd[0, 0::2] = (121, 122)
    sd[0, 1::2] = (122, 122)
    W = {"w_gate": code((1, 64, 64)), "w_up": code((1, 64, 64)), "w_down": code((1, 64, 64)),
         "s_gate": np.tile(np.array([121, 120], np.uint8), (1, 64, 1)),
         "s_up": np.tile(np.array([122, 121], np.uint8), (1, 64, 1)), "s_down": sd,
         "ws_gate": None, "ws_up": None, "ws_down": None, "ss_gate": None, "ss_up": None, "ss_down": None}
    x = np.full((1, 64), 0x3F80, np.uint16)  # bf16 1.0
    for aq, tag in ((True, "on"), (False, "off")):
        y = orc.forward_tokens_mx(cfg, orc.WeightsMX(W), x, [[0]], [[0.5]], act_quant=aq)[0]
        np.testing.assert_allclose(y[0::2], g[f"{tag}_even"], rtol=1e-14)
        np.testing.assert_allclose(y[1::2], g[f"{tag}_odd"], rtol=1e-14)


def _deq(codes, scales):
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)
    s = torch.exp2(torch.from_numpy(scales.astype(np.float64)) - 127).repeat_interleave(32, dim=-1)
    return c * s


def test_mx_layer_against_torch_fp64(orc):
    cfg = MoEConfig(256, 128, 4, 2, 1, 2, 1.0, 1)
    W = {k: (None if v is None else v.numpy()) for k, v in make_weights_mx(cfg, 3).items()}
    x = make_tokens(cfg, 5, 4)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    ids = np.array([[0, 3], [1, 2], [2, 2 - 2], [3, 1], [0, 1]], np.int32)
    w = np.array([[0.7, 0.2], [0.5, 0.5], [1.5, 0.1], [0.25, 2.0], [0.0, 1.0]])
    got = orc.forward_tokens_mx(cfg, orc.WeightsMX(W), xb, ids, w)

    def mlp(xh, wg, sg, wu, su, wd, sd):
        gg, uu = _deq(wg, sg) @ xh, _deq(wu, su) @ xh
        a = (gg / (1 + torch.exp(-gg)) * uu).numpy()
        qa, sa = orc.quant_rows_mx(a[None, :])
        ah = _deq(qa, sa)[0]
        return _deq(wd, sd) @ ah

    for t in range(5):
        qx, sx = orc.quant_rows_mx(x[t].double().numpy()[None, :])
        xh = _deq(qx, sx)[0]
        ref = sum(w[t, j] * mlp(xh, W["w_gate"][ids[t, j]], W["s_gate"][ids[t, j]], W["w_up"][ids[t, j]],
                                W["s_up"][ids[t, j]], W["w_down"][ids[t, j]], W["s_down"][ids[t, j]])
                  for j in range(2))
        ref = ref + mlp(xh, W["ws_gate"], W["ss_gate"], W["ws_up"], W["ss_up"], W["ws_down"], W["ss_down"])
        np.testing.assert_allclose(got[t], ref.numpy(), rtol=1e-10, atol=1e-12)
