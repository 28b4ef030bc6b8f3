"""Pins for the oracle's element formats and quantisation rule (CPU only).

Each check ties the oracle to something other than itself: the published format
tables (tests/golden/, with their citations), PyTorch's own fp8 / e8m0 / bf16
conversions, closed forms written independently with math.ldexp, and brute force.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            rows.append((int(c, 0), float(v)))
    return rows


def _same(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(
        np.nan_to_num(a), np.nan_to_num(b)) and np.array_equal(
        np.signbit(a[~np.isnan(a)]), np.signbit(b[~np.isnan(b)]))


def test_e2m1_matches_spec_table():
    rows = _read_table("e2m1_values.txt")
    codes = [c for c, _ in rows]
    assert _same(o.e2m1_decode(codes), [v for _, v in rows])


def test_e2m1_times_e8m0_exhaustive():
    """16 codes x 255 finite scale bytes against (-1)^s * table[m] * 2^(b-127)."""
    table = dict(_read_table("e2m1_values.txt"))
    codes = np.repeat(np.arange(16), 255)
    scales = np.tile(np.arange(255), 16)
    got = o.e2m1_decode(codes) * o.e8m0_decode(scales)
    want = [math.ldexp(table[c], int(b) - 127) for c, b in zip(codes, scales)]
    assert _same(got, want)


def test_e8m0_matches_spec_and_torch():
    rows = _read_table("e8m0_landmarks.txt")
    assert _same(o.e8m0_decode([c for c, _ in rows]), [v for _, v in rows])
    allc = torch.arange(256, dtype=torch.uint8)
    ref = allc.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert _same(o.e8m0_decode(np.arange(256)), ref)


def test_e4m3_decode_all_codes():
    rows = _read_table("e4m3_landmarks.txt")
    assert _same(o.e4m3_decode([c for c, _ in rows]), [v for _, v in rows])
    allc = torch.arange(256, dtype=torch.uint8)
    ref = allc.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert _same(o.e4m3_decode(np.arange(256)), ref)


def test_e4m3_encode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    assert np.array_equal(o.e4m3_encode(o.e4m3_decode(codes)), codes)


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_midpoints_ties_to_even():
    pos = o.e4m3_decode(np.arange(0x7F))
    mids = (pos[:-1] + pos[1:]) / 2.0          # exact in float32 too
    got = o.e4m3_encode(np.concatenate([mids, -mids]))
    assert np.array_equal(got, _torch_e4m3(np.concatenate([mids, -mids])))
    # explicit: the even code wins every tie
    up = np.arange(1, 0x7F)
    even = np.where(up % 2 == 0, up, up - 1)
    assert np.array_equal(o.e4m3_encode(mids), even)


def test_e4m3_encode_random_against_torch():
    rng = np.random.default_rng(1)
    mag = np.ldexp(rng.uniform(1, 2, 1_000_000), rng.integers(-12, 9, 1_000_000))
    v = (mag * rng.choice([-1, 1], 1_000_000)).astype(np.float32)
    v = v[np.abs(v) <= 448]
    assert np.array_equal(o.e4m3_encode(v.astype(np.float64)), _torch_e4m3(v))


def test_e4m3_encode_signed_zero_and_saturation():
    assert o.e4m3_encode([-0.0])[0] == 0x80
    assert o.e4m3_encode([0.0])[0] == 0x00
    assert o.e4m3_encode([-1e-12])[0] == 0x80
    assert o.e4m3_encode([1000.0])[0] == 0x7E
    assert o.e4m3_encode([-1000.0])[0] == 0xFE


def test_bf16_round_against_torch_for_fp32_inputs():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(200_000) * np.ldexp(1.0, rng.integers(-30, 30, 200_000))
         ).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o.bf16_round(v.astype(np.float64)), want)


def test_bf16_round_float64_is_nearest_ties_even():
    """float64 inputs: brute force against the two bf16 neighbours (no double rounding)."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal(20000) * np.ldexp(1.0, rng.integers(-20, 20, 20000))
    # add exact ties and values 1 float64-ulp away from ties
    base = o.bf16_round(v)
    _, p = np.frexp(base)
    half = np.ldexp(1.0, p - 9)
    ties = base + half
    v = np.concatenate([v, ties, np.nextafter(ties, np.inf), np.nextafter(ties, -np.inf)])
    got = o.bf16_round(v)
    f32 = v.astype(np.float32)
    b = (f32.view(np.uint32) >> 16).astype(np.uint32)
    lo = ((b << 16).view(np.float32)).astype(np.float64)
    hi = (((b + 1) << 16).view(np.float32)).astype(np.float64)
    lo2 = ((((b - 1) << 16)).view(np.float32)).astype(np.float64)
    cands = np.stack([lo2, lo, hi], axis=1)
    d = np.abs(cands - v[:, None])
    best = d.min(axis=1)
    assert np.all(np.abs(got - v) == best)
    tie = (d == best[:, None]).sum(axis=1) > 1
    gb = (got[tie].astype(np.float32).view(np.uint32) >> 16)
    assert np.all(gb % 2 == 0)


def test_scale_exponent_brute_force_minimal():
    """Every bf16 value in [2^-20, 2^20]: e is the smallest integer with
    amax <= 448 * 2^e (exact comparisons in float64)."""
    lo = np.array([2.0 ** -20], dtype=np.float32).view(np.uint32)[0] >> 16
    hi = np.array([2.0 ** 20], dtype=np.float32).view(np.uint32)[0] >> 16
    bits = np.arange(lo, hi + 1, dtype=np.uint32) << 16
    amax = bits.view(np.float32).astype(np.float64)
    e = o.scale_exponent(amax)
    assert np.all(amax <= 448.0 * np.ldexp(1.0, e))
    assert np.all(amax > 448.0 * np.ldexp(1.0, e - 1))


def test_scale_exponent_landmarks():
    assert o.scale_exponent([448.0])[0] == 0
    assert o.scale_exponent([448.0 * (1 + 2 ** -7)])[0] == 1
    assert o.scale_exponent([1.75])[0] == -8
    assert o.scale_exponent([1.0])[0] == -8
    assert o.scale_exponent([1.7578125])[0] == -7
    assert o.scale_exponent([0.0])[0] == 0
    assert o.scale_exponent([1e-45])[0] == -127


def test_quant_rows_properties():
    rng = np.random.default_rng(4)
    x = o.bf16_round(rng.standard_normal((16, 512)) * np.ldexp(1.0, rng.integers(-10, 10, (16, 1))))
    x[3, :128] = 0.0
    x[5, 128:256] = -0.0
    q, s = o.quant_rows(x)
    assert s.shape == (16, 4) and q.shape == (16, 512)
    assert np.all(s[3, 0] == 127) and np.all(q[3, :128] == 0)
    assert np.all(q[5, 128:256] == 0x80)
    # every code is a nearest E4M3 value of x * 2^-e
    e = s.astype(np.int64) - 127
    y = np.ldexp(x.reshape(16, 4, 128), -e[:, :, None]).reshape(16, 512)
    assert np.abs(y).max() <= 448
    dec = o.e4m3_decode(q)
    pos = o.e4m3_decode(np.arange(0x7F))
    nearest = np.abs(pos[None, :] - np.abs(y).reshape(-1, 1)).min(axis=1).reshape(y.shape)
    assert np.all(np.abs(np.abs(dec) - np.abs(y)) == nearest)
    # the block maximum maps into the top binade (scale is minimal): |amax*2^-e| > 224
    amax = np.abs(y.reshape(16, 4, 128)).max(axis=2)
    assert np.all((amax > 224) | (amax == 0))


def test_quant_act_block_with_amax_448_is_identity_scale():
    """A block whose amax is exactly 448 keeps scale 2^0 and exact codes."""
    vals = np.array([448.0, -448.0, 1.0, 2.0, 0.5, -0.25] + [0.0] * 122)
    bits = o.f64_to_bf16_bits(vals)[None, :]
    q, s = o.quant_act(bits)
    assert s[0, 0] == 127
    assert list(q[0, :6]) == [0x7E, 0xFE, 0x38, 0x40, 0x30, 0xA8]
