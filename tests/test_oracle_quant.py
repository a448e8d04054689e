"""Pins for oracle.quant: Q_2(.; c, 128), fp16 meta, 2-bit packing."""
import json
import os

import numpy as np
import pytest

from oracle import quant
from conftest import GOLDEN


def _golden():
    with open(os.path.join(GOLDEN, "quant_examples.json")) as f:
        return json.load(f)["examples"]


def _example_input(ex):
    if ex.get("ramp_mod4"):
        return ex["offset"] + (np.arange(128) % 4).astype(np.float64)
    x = np.full(128, ex["fill"], dtype=np.float64)
    x[: len(ex["pattern"])] = ex["pattern"]
    return x


@pytest.mark.parametrize("ex", _golden(), ids=lambda e: e["name"])
def test_hand_worked_groups(ex):
    x = _example_input(ex)
    codes, s, z = quant.quantize_groups(x[None], ex["clip"])
    assert int(quant.fp16_bits(s)[0]) == ex["scale_bits"]
    assert int(quant.fp16_bits(z)[0]) == ex["zero_bits"]
    assert codes[0, :8].tolist() == ex["codes_head"]
    assert quant.pack_codes(codes)[0].tobytes().hex() == ex["packed"]


def test_fp16_rounding_is_direct_round_half_even():
    # 1 + 2^-11 is the midpoint between 1 and 1 + 2^-10: ties go to even (1.0)
    assert quant.fp16_rne(1 + 2 ** -11) == 1.0
    # slightly above the midpoint must round up; rounding through float32 first would not
    assert quant.fp16_rne(1 + 2 ** -11 + 2 ** -40) == 1 + 2 ** -10
    assert int(quant.fp16_bits(quant.fp16_rne(1 / 3))) == 0x3555


def _random_groups(n, seed):
    g = np.random.default_rng(seed)
    x = g.standard_normal((n, 128)) * g.uniform(0.01, 30, (n, 1)) + g.normal(0, 5, (n, 1))
    x[::7, 3] += 40.0  # outliers
    return x


@pytest.mark.parametrize("clip", [1.0, 0.95, 0.8, 0.5])
def test_codes_equal_nearest_level_brute_force(clip):
    x = _random_groups(400, 1)
    codes, s, z = quant.quantize_groups(x, clip)
    levels = z[:, None, None] + s[:, None, None] * np.arange(4)[None, None, :]  # [n,1,4]
    dist = np.abs(x[:, :, None] - levels)
    brute = dist.argmin(axis=-1)
    assert np.array_equal(codes, brute)


@pytest.mark.parametrize("clip", [1.0, 0.9])
def test_dequantized_values_lie_on_the_four_level_grid(clip):
    x = _random_groups(200, 2)
    codes, s, z = quant.quantize_groups(x, clip)
    xh = quant.dequantize_groups(codes, s, z)
    grid = z[:, None, None] + s[:, None, None] * np.arange(4)[None, None, :]
    assert np.all(np.min(np.abs(xh[:, :, None] - grid), axis=-1) == 0.0)
    assert codes.max() <= 3 and codes.min() >= 0


def test_error_bound_clip_one():
    x = _random_groups(300, 3)
    codes, s, z = quant.quantize_groups(x, 1.0)
    xh = quant.dequantize_groups(codes, s, z)
    lo = x.min(axis=1)
    hi = x.max(axis=1)
    bound = s / 2 + np.abs(lo - z) + 3 * np.abs((hi - lo) / 3 - s)
    assert np.all(np.abs(x - xh).max(axis=1) <= bound * (1 + 1e-12) + 1e-15)


def test_min_and_max_land_on_end_levels_for_clip_one():
    x = _random_groups(100, 4)
    codes, _, _ = quant.quantize_groups(x, 1.0)
    assert np.all(codes[np.arange(100), x.argmin(axis=1)] == 0)
    assert np.all(codes[np.arange(100), x.argmax(axis=1)] == 3)


def test_degenerate_group_reconstructs_its_value():
    x = np.full((2, 128), -7.25)
    codes, s, z = quant.quantize_groups(x, 0.9)
    assert np.all(codes == 0) and np.all(s == 0)
    assert np.all(quant.dequantize_groups(codes, s, z) == quant.fp16_rne(0.9 * -7.25))


def test_identity_rotation_is_plain_int2():
    # Eq. 4 with R = I: D_{I,c}(x) = Q_2(x; c)
    x = _random_groups(50, 5)
    assert np.array_equal(quant.rotated_quant_dequant(x, np.eye(128), 0.9), quant.quant_dequant(x, 0.9))


def test_pack_unpack_round_trip_and_bit_order():
    g = np.random.default_rng(6)
    c = g.integers(0, 4, (10, 128)).astype(np.uint8)
    p = quant.pack_codes(c)
    assert p.shape == (10, 32)
    assert np.array_equal(quant.unpack_codes(p), c)
    one = np.zeros(128, np.uint8)
    one[5] = 3  # channel 5 -> byte 1, bits 2..3
    pb = quant.pack_codes(one)
    assert pb[1] == 0b00001100 and pb.sum() == 12


def test_near_boundary_flags_midpoints_only():
    s = np.array([0.5])
    z = np.array([-1.0])
    x = np.array([[-1.0 + 0.25, -1.0 + 0.5 * 0.5 + 1e-9, 0.0, -1.0 + 0.75]])
    hit = quant.near_boundary(np.pad(x, ((0, 0), (0, 124)), constant_values=-1.0), s, z)
    assert hit[0, :4].tolist() == [True, True, False, True]


def test_group_near_fp16_tie():
    x = np.zeros((2, 128))
    x[0, 0] = 3 * (1 + 2 ** -11)  # (hi - lo)/3 = 1 + 2^-11, an fp16 midpoint
    x[1, 0] = 3.0
    flags = quant.group_near_fp16_tie(x, 1.0)
    assert flags.tolist() == [True, False]
