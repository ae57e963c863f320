"""Pins of the oracle's number formats: e4m3 (OCP 8-bit FP, E4M3), bf16 and the
fp32 exponential used by SwiGLU.  Nothing here needs a GPU."""

import math
import struct

import numpy as np
import pytest
import torch

import oracle


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def f32_from_bits(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


# ---------------------------------------------------------------- e4m3 -----

def test_e4m3_spec_values():
    # Values fixed by the OCP FP8 E4M3 definition (bias 7, no infinities).
    t = oracle.e4m3_table()
    assert t[0x00] == 0.0 and math.copysign(1, t[0x80]) < 0
    assert t[0x01] == 2.0 ** -9          # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x38] == 1.0
    assert t[0x39] == 1.125
    assert t[0x7E] == 448.0              # largest finite
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert t[0xFE] == -448.0


def test_e4m3_decode_matches_torch():
    # torch's float8_e4m3fn decode is an independent library routine.
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = codes.to(torch.float64).numpy()
    t = oracle.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(t))
    assert np.array_equal(ref[~nan], t[~nan])


def test_e4m3_roundtrip_all_codes():
    t = oracle.e4m3_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.f32_to_e4m3(t[c]) == c, hex(c)


def test_e4m3_monotone_and_ties_to_even():
    t = oracle.e4m3_table()
    pos = t[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)
    for c in range(0x00, 0x7E):
        lo, hi = t[c], t[c + 1]
        mid = (lo + hi) / 2.0          # exact in fp32: at most 5 significant bits
        assert np.float32(mid) == mid
        even = c if (c & 1) == 0 else c + 1
        assert oracle.f32_to_e4m3(mid) == even
        assert oracle.f32_to_e4m3(-mid) == (even | 0x80)
        below = np.nextafter(np.float32(mid), np.float32(0))
        above = np.nextafter(np.float32(mid), np.float32(1000))
        assert oracle.f32_to_e4m3(below) == c
        assert oracle.f32_to_e4m3(above) == c + 1


def test_e4m3_saturation_and_signed_zero():
    assert oracle.f32_to_e4m3(448.0) == 0x7E
    assert oracle.f32_to_e4m3(449.0) == 0x7E
    assert oracle.f32_to_e4m3(1e30) == 0x7E
    assert oracle.f32_to_e4m3(float("inf")) == 0x7E
    assert oracle.f32_to_e4m3(-1e30) == 0xFE
    assert oracle.f32_to_e4m3(0.0) == 0x00
    assert oracle.f32_to_e4m3(-0.0) == 0x80
    # below half the smallest subnormal: rounds to zero, sign kept
    assert oracle.f32_to_e4m3(2.0 ** -11) == 0x00
    assert oracle.f32_to_e4m3(-(2.0 ** -11)) == 0x80
    # exactly half the smallest subnormal ties to the even code 0
    assert oracle.f32_to_e4m3(2.0 ** -10) == 0x00


def test_e4m3_encode_matches_torch_in_range():
    # torch rounds to nearest-even but turns values above 464 into NaN, so
    # the comparison is restricted to |v| < 464 where both must agree.
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.uniform(-463.9, 463.9, 20000),
        rng.standard_normal(20000) * 0.01,
        rng.standard_normal(20000) * 1e-3,
        np.exp(rng.uniform(-14, 6, 20000)) * rng.choice([-1, 1], 20000),
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.f32_to_e4m3(x) for x in v], np.uint8)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- bf16 -----

def _bf16_candidates(d: float):
    """Brute force: the two bf16 values around d and the nearest-even pick."""
    f = np.float32(d)  # nearby float; candidates are its bf16 truncations +-1
    u = f32_bits(float(f)) & 0xFFFF0000
    cands = [(u + k * 0x10000) & 0xFFFFFFFF for k in (-2, -1, 0, 1, 2)]
    best = None
    for c in cands:
        v = f32_from_bits(c)
        if math.isnan(v) or math.isinf(v):
            continue
        err = abs(v - d)
        key = (err, (c >> 16) & 1)
        if best is None or key < best[0]:
            best = (key, c >> 16)
    return best[1]


def test_bf16_round_brute_force():
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.standard_normal(3000), rng.standard_normal(1000) * 1e-30,
                           rng.uniform(-1e4, 1e4, 1000)])
    # exact ties: a bf16 value plus half its quantum
    ties = []
    for x in rng.standard_normal(500):
        b = f32_bits(float(np.float32(x))) & 0xFFFF0000
        lo, hi = f32_from_bits(b), f32_from_bits(b + 0x10000)
        ties.append((lo + hi) / 2)
    vals = np.concatenate([vals, np.array(ties)])
    got = oracle.f64_to_bf16(vals)
    for d, g in zip(vals, got):
        assert int(g) == _bf16_candidates(float(d)), d


def test_bf16_matches_torch_from_fp32():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(v.astype(np.float64)), ref)


# ------------------------------------------------------------ fp32 exp -----

def _ulp_dist(a: float, b: float) -> int:
    ia, ib = f32_bits(a), f32_bits(b)
    if ia >> 31:
        ia = 0x80000000 - ia
    if ib >> 31:
        ib = 0x80000000 - ib
    return abs(ia - ib)


def test_exp_f32_accuracy_sweep():
    rng = np.random.default_rng(4)
    xs = np.concatenate([rng.uniform(-87.0, 88.5, 20000), rng.uniform(-1, 1, 5000),
                         np.linspace(-20, 20, 4001)]).astype(np.float32)
    worst = 0
    for x in xs:
        ref = float(np.float32(math.exp(float(x))))  # correctly rounded to fp32 (almost always)
        worst = max(worst, _ulp_dist(oracle.exp_f32(x), ref))
    assert worst <= 2


def test_exp_f32_special_values():
    assert oracle.exp_f32(0.0) == 1.0
    assert oracle.exp_f32(-0.0) == 1.0
    assert oracle.exp_f32(89.0) == float("inf")
    assert oracle.exp_f32(-104.0) == 0.0
    # subnormal results: within one quantum (2^-149) of the true value
    for x in (-90.0, -95.5, -100.0, -103.0):
        assert abs(oracle.exp_f32(x) - math.exp(x)) <= 2.0 ** -149


def test_silu_f32_against_f64():
    rng = np.random.default_rng(5)
    for z in np.concatenate([rng.standard_normal(5000) * 4, [0.0, -80.0, 80.0, -100.0, 100.0]]).astype(np.float32):
        z = float(z)
        ref = z / (1.0 + math.exp(-z))
        got = oracle.silu_f32(z)
        assert abs(got - ref) <= 4e-7 * abs(ref) + 1e-37, z
