"""Pins for the oracle's NVFP4 weight format (f3; GB10 "Optimization progress
report", Optimization 05, native NVFP4 MoE).  CPU only.

NVFP4 as read here: E2M1 codes (two per byte, even K index in the low nibble), one FP8
E4M3 scale per 16 consecutive K elements, and an fp32 scale per weight tensor (W13:
one for the gate rows, one for the up rows).  Each check ties the oracle to
something other than itself: the OCP E2M1 table (tests/golden/e2m1_values.txt), an
E4M3 closed form written here with math.ldexp, PyTorch's float8_e4m3fn conversion,
integer arithmetic, and the MXFP4 path where the two formats coincide."""

import math
import os

import numpy as np
import torch

from gen import inputs as gi
from oracle import moe_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_table():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                vals[int(c, 0)] = float(v)
    return [vals[c] for c in range(16)]


def _e4m3_closed_form(b):
    """E4M3 ("FN") byte -> value, from its bit fields: sign, 4-bit exponent (bias 7),
    3-bit mantissa; exponent 0 subnormal; S.1111.111 NaN."""
    s = -1.0 if b & 0x80 else 1.0
    e, m = (b >> 3) & 0xF, b & 0x7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m, -9)
    return s * math.ldexp(8 + m, e - 10)


def _codes_row_all_16():
    """One row of 16 K elements holding the codes 0..15 in K order."""
    c = np.arange(16, dtype=np.uint8)
    return (c[0::2] | (c[1::2] << 4))[None, :]


def test_nvfp4_dequant_exhaustive_closed_form():
    """Every E2M1 code under every one of the 256 E4M3 scale bytes."""
    e2m1 = _e2m1_table()
    codes = np.repeat(_codes_row_all_16(), 256, axis=0)          # [256, 8]
    scales = np.arange(256, dtype=np.uint8)[:, None]              # [256, 1]
    got = o.nvfp4_dequant(codes, scales)
    want = np.array([[e2m1[c] * _e4m3_closed_form(b) for c in range(16)]
                     for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_nvfp4_dequant_against_torch_e4m3():
    e2m1 = np.array(_e2m1_table())
    rng = np.random.default_rng(3)
    N, K = 64, 256
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, size=(N, K // 16), dtype=np.uint8)  # finite, signed below
    scales[::3] |= 0x80
    s_t = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nib = np.empty((N, K), np.int64)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = codes >> 4
    want = e2m1[nib] * np.repeat(s_t, 16, axis=1)
    assert np.array_equal(o.nvfp4_dequant(codes, scales), want)


def test_nvfp4_scale_block_is_16_elements():
    """Changing one scale byte changes exactly its 16 K elements, by the scale ratio."""
    rng = np.random.default_rng(4)
    N, K = 8, 128
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = np.full((N, K // 16), 0x38, np.uint8)  # 1.0
    base = o.nvfp4_dequant(codes, scales)
    for n0, b0 in ((0, 0), (3, 5), (7, 7)):
        s2 = scales.copy()
        s2[n0, b0] = 0x40  # 2.0
        w = o.nvfp4_dequant(codes, s2)
        mask = np.zeros((N, K), bool)
        mask[n0, 16 * b0:16 * b0 + 16] = True
        assert np.array_equal(w[~mask], base[~mask])
        assert np.array_equal(w[mask], 2.0 * base[mask])


def test_nvfp4_tensor_scale_per_row_segment():
    rng = np.random.default_rng(5)
    N, K = 12, 64
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.integers(0x20, 0x48, size=(N, K // 16), dtype=np.uint8)
    base = o.nvfp4_dequant(codes, scales)
    gs = np.array([0.75, 3.0], np.float32)
    w = o.nvfp4_dequant(codes, scales, gs)
    assert np.array_equal(w[:6], 0.75 * base[:6]) and np.array_equal(w[6:], 3.0 * base[6:])
    assert np.array_equal(o.nvfp4_dequant(codes, scales, 0.5), 0.5 * base)


def test_nvfp4_equals_mxfp4_when_scales_agree():
    """NVFP4 with E4M3 block scales 2^e and MXFP4 with E8M0 scales 2^e (each 32-block
    of MXFP4 = two 16-blocks with the same scale) decode to the same matrix."""
    rng = np.random.default_rng(6)
    N, K = 16, 256
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    e = rng.integers(-4, 1, size=(N, K // 32))
    mx_s = (e + 127).astype(np.uint8)
    nv_s = np.repeat(((e + 7) << 3).astype(np.uint8), 2, axis=1)  # E4M3 2^e, e in [-4, 0]
    assert np.array_equal(o.nvfp4_dequant(codes, nv_s), o.mxfp4_dequant(codes, mx_s))


def _int_act(rows, K, seed):
    codes = gi.integer_codes((rows, K), gi.E4M3_INTEGER_CODES, seed, "cpu", "act").numpy()
    return codes, np.full((rows, K // 128), 127, np.uint8)


def test_nvfp4_grouped_gemm_exact_integers():
    """Integer-valued activations x integer E2M1 codes x integer E4M3 block scales and
    power-of-two tensor scales: every y is the exact integer dot product, computed
    here with Python integers from the code bytes."""
    rng = np.random.default_rng(7)
    e2m1 = _e2m1_table()
    G, N, K = 2, 12, 256
    offsets = np.array([0, 5, 9], np.int32)
    aq, asc = _int_act(9, K, 8)
    xv = o.e4m3_decode(aq).astype(np.int64)
    int_codes = [c for c in range(16) if e2m1[c] == int(e2m1[c])]
    nib = rng.choice(int_codes, size=(G, N, K))
    wq = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    # block scales 1, 2, 3 (0x38, 0x40, 0x44) and tensor scales 2^-1 / 2
    ws = rng.choice([0x38, 0x40, 0x44], size=(G, N, K // 16)).astype(np.uint8)
    gsc = np.array([[0.5, 2.0], [2.0, 0.5]], np.float32)
    y = o.grouped_gemm(aq, asc, offsets, wq, ws, fmt="nvfp4", w_global=gsc)
    sval = {0x38: 1, 0x40: 2, 0x44: 3}
    for g in range(G):
        for r in range(offsets[g], offsets[g + 1]):
            for n in range(N):
                acc = sum(int(xv[r, k]) * int(e2m1[nib[g, n, k]]) * sval[ws[g, n, k // 16]]
                          for k in range(K))
                exact = acc * float(gsc[g, n // (N // 2)])
                assert y[r, n] == float(o.bf16_round(np.float64(exact)))


def test_dense_unrouted_equals_routed_nvfp4():
    d = gi.Dims(T=24, H=256, I=128, E=6, k=2, has_shared=1)
    t = gi.custom_layer(d, seed=3)
    nv = gi.nvfp4_layer_weights(d, seed=3)
    x = t["x"].view(torch.int16).numpy().view(np.uint16)
    lg = t["logits"].numpy()
    a = o.moe_forward(x, lg, d.k, nv["w13"].numpy(), nv["w13_s"].numpy(), nv["w2"].numpy(),
                      nv["w2_s"].numpy(), d.has_shared, "nvfp4", nv["w13_gs"].numpy(),
                      nv["w2_gs"].numpy())["out"]
    b = o.dense_unrouted_forward(x, lg, d.k, nv["w13"].numpy(), nv["w13_s"].numpy(),
                                 nv["w2"].numpy(), nv["w2_s"].numpy(), d.has_shared, "nvfp4",
                                 nv["w13_gs"].numpy(), nv["w2_gs"].numpy())
    assert np.array_equal(a, b)
    assert np.all(np.isfinite(a)) and np.any(a != 0)
