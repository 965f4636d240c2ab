"""Pins of the oracle's stage M (RMSNorm in front of the router) and its bf16 rounding.

Stage M of the DSV2-236B-MegaKernel stage flowchart (MoE subgraph), the hidden
state normalised and scaled by gamma before the router: x = h / sqrt(mean(h^2) + eps) * gamma per token row, rounded once to
bf16. Pinned by a hand-worked row (tests/golden/rmsnorm_hand.txt), closed forms
(a constant row normalises to +-1), invariances the definition implies (scaling h by
a power of two, gamma by a power of two), torch's float32 -> bf16 conversion for the
rounding, and a torch fp64 evaluation of the formula.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rmsnorm_hand.txt")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_from_float(v) -> np.ndarray:
    return _bits(torch.tensor(np.asarray(v, np.float32)))


def _golden():
    vals = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_round_bf16_matches_torch_on_float32_values(orc):
    # a float32 value rounds to bf16 in one step either way, so the oracle's direct
    # fp64 rounding must agree with torch's float32 -> bf16 conversion (RNE)
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-3).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        np.array([1e-40, -3e-39, 1.17549435e-38, 3.3895314e38, -3.3895314e38], np.float32),
    ])
    got = orc.round_bf16(v.astype(np.float64))
    assert np.array_equal(got, _bf16_from_float(v))


def test_round_bf16_ties_go_to_even(orc):
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even significand (1.0) wins;
    # 1 + 3 * 2^-8 lies between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    got = orc.round_bf16([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** 128, 3.0])
    assert got.tolist() == [0x3F80, 0x3F82, 0xBF80, 0x7F80, 0x4040]


def test_rmsnorm_hand_worked_row(orc):
    g = _golden()
    h = np.zeros(128, np.float32)
    h[0], h[1] = 3.0, 4.0
    hb = _bf16_from_float(h)[None, :]
    one = _bf16_from_float(np.ones(128, np.float32))
    for eps in (0.0, 1e-6):
        x = orc.rmsnorm(hb, one, eps)
        assert x[0, 0] == _bf16_from_float([g["x0"]])[0]
        assert x[0, 1] == _bf16_from_float([g["x1"]])[0]
        assert not x[0, 2:].any()
    gam = np.ones(128, np.float32)
    gam[0] = 0.5
    x = orc.rmsnorm(hb, _bf16_from_float(gam), 0.0)
    assert x[0, 0] == _bf16_from_float([g["x0_gamma_half"]])[0]


@pytest.mark.parametrize("c", [0.75, -3.0, 1e-3, 250.0])
def test_rmsnorm_constant_row_is_unit(orc, c):
    H = 256
    h = _bf16_from_float(np.full((2, H), c, np.float32))
    x = orc.rmsnorm(h, _bf16_from_float(np.ones(H, np.float32)), 0.0)
    assert np.all(x == _bf16_from_float([np.sign(c)])[0])


def test_rmsnorm_zero_row_with_eps(orc):
    H = 128
    x = orc.rmsnorm(np.zeros((1, H), np.uint16), _bf16_from_float(np.ones(H, np.float32)), 1e-6)
    assert not x.any()


def test_rmsnorm_invariances(orc):
    rng = np.random.default_rng(3)
    H = 512
    h = rng.standard_normal((4, H)).astype(np.float32)
    gam = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    hb, gb = _bf16_from_float(h), _bf16_from_float(gam)
    base = orc.rmsnorm(hb, gb, 0.0)
    # scaling h by a power of two cancels exactly
    for j in (-5, 3):
        assert np.array_equal(orc.rmsnorm(_bf16_from_float(h * 2.0 ** j), gb, 0.0), base)
    # scaling gamma by a power of two scales every (rounded) output exactly
    x4 = orc.rmsnorm(hb, _bf16_from_float(gam * 4), 0.0)
    as_f = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(as_f(x4), as_f(base) * 4)
    # permuting the channels permutes the output
    perm = rng.permutation(H)
    assert np.array_equal(orc.rmsnorm(hb[:, perm], gb[perm], 0.0), base[:, perm])


def test_rmsnorm_against_torch_fp64(orc):
    rng = np.random.default_rng(11)
    T, H, eps = 6, 5120, 1e-6
    hb = _bf16_from_float(rng.standard_normal((T, H)) * 2)
    gb = _bf16_from_float(1 + 0.2 * rng.standard_normal(H))
    to_f64 = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double()
    hh, gg = to_f64(hb), to_f64(gb)
    ref = hh / torch.sqrt((hh * hh).mean(dim=1, keepdim=True) + eps) * gg
    x, exact = orc.rmsnorm(hb, gb, eps, return_exact=True)
    np.testing.assert_allclose(exact, ref.numpy(), rtol=1e-13, atol=0)
    # rounding: torch converts fp64 -> fp32 -> bf16 (two roundings); the single rounding
    # may differ from it only where the fp64 value sits within fp32 precision of a tie
    tor = _bits(ref.float())
    diff = x != tor
    a = np.abs(ref.numpy())
    q = np.exp2(np.floor(np.log2(a)) - 7)
    dist = np.abs(a / q - np.floor(a / q) - 0.5) * q / a
    assert np.all(dist[diff] < 2.0 ** -23)
