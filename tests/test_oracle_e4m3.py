"""Pins of the oracle's FP8 E4M3 decode/encode and its activation quantisation.

The E4M3 format (OCP FP8, "E4M3FN": bias 7, no infinities, max 448) is what the
pages' "per-128 block-scaled FP8" weights are stored in (DSV2-236B-MegaKernel,
README "Results" and quant/fp8_block_quant.py in its "Layout"). Pinned against
torch's float8_e4m3fn conversion (a library routine) and hand-worked values.
"""
import numpy as np
import pytest
import torch


def test_decode_all_256_codes_match_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign bit
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x7E, 448.0),
    (0xB8, -1.0), (0xFE, -448.0),
])
def test_decode_hand_values(orc, code, value):
    assert orc.e4m3_decode(np.array([code], np.uint8))[0] == value


def test_encode_roundtrips_every_finite_code(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_decode(codes)
    assert np.array_equal(orc.e4m3_encode(vals), codes)


def test_encode_matches_torch_rne_in_range(orc):
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.uniform(-448, 448, 4000),
        rng.normal(0, 1, 4000),
        rng.normal(0, 1e-2, 2000),   # subnormal range
        rng.normal(0, 30, 2000),
    ])
    ours = orc.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("value,code", [
    (1.0625, 0x38),        # halfway 1.0 / 1.125 -> even mantissa (1.0)
    (1.1875, 0x3A),        # halfway 1.125 / 1.25 -> 1.25 (even)
    (2.0 ** -10, 0x00),    # halfway 0 / smallest subnormal -> 0
    (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 / 2^-8 -> 2^-8 (even)
    (-1.0625, 0xB8),
    (464.0, 0x7E),         # beyond the grid saturates to 448
    (1e9, 0x7E),
    (-1e9, 0xFE),
    (float("nan"), 0x7F),
])
def test_encode_ties_and_saturation(orc, value, code):
    assert orc.e4m3_encode(np.array([value]))[0] == code


# ----------------------------------------------------- activation quantisation
def _block(amax, n=128, seed=0):
    rng = np.random.default_rng(seed)
    v = rng.uniform(-amax, amax, n)
    v[5] = amax
    return v


@pytest.mark.parametrize("amax,scale", [
    (448.0, 1.0),            # exactly representable at scale 1
    (449.0, 2.0),            # just above -> next power of two
    (1.0, 2.0 ** -8),        # 448 * 2^-9 = 0.875 < 1 <= 1.75 = 448 * 2^-8
    (0.875, 2.0 ** -9),      # the boundary itself is inclusive
    (0.8750001, 2.0 ** -8),
    (896.0, 2.0),
    (3.0, 2.0 ** -7),
])
def test_act_scale_is_smallest_power_of_two_covering_amax(orc, amax, scale):
    q, s = orc.quant_rows(_block(amax)[None, :])
    assert s[0, 0] == scale
    # the block maximum lands on the grid's top decade, never above 448
    dq = orc.e4m3_decode(q[0]) * s[0, 0]
    assert np.nanmax(np.abs(dq)) <= 448 * scale


def test_act_quant_zero_block(orc):
    q, s = orc.quant_rows(np.zeros((1, 256)))
    assert np.all(q == 0) and np.all(s == 1.0)


def test_act_quant_is_identity_on_grid_values(orc):
    # values already on the E4M3 grid times 2^-3, with the block max = 448 * 2^-3
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 0x7E, 128).astype(np.uint8) | (rng.integers(0, 2, 128).astype(np.uint8) << 7)
    codes[0] = 0x7E
    v = orc.e4m3_decode(codes) * 2.0 ** -3
    q, s = orc.quant_rows(v[None, :])
    assert s[0, 0] == 2.0 ** -3
    assert np.array_equal(orc.e4m3_decode(q[0]) * s[0, 0], v)


def test_act_quant_codes_match_torch_cast_of_scaled_values(orc):
    rng = np.random.default_rng(3)
    v = rng.normal(0, 1, (16, 512)) * rng.uniform(1e-3, 10, (16, 1))
    q, s = orc.quant_rows(v)
    scaled = v / np.repeat(s, 128, axis=1)
    ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    # blocks are independent: each block's scale only depends on its own max
    amax = np.abs(v).reshape(16, 4, 128).max(-1)
    assert np.all(amax <= 448 * s) and np.all(amax > 224 * s)
