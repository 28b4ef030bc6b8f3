"""Pins of the oracle's router gate projection (logits = x . W_g^T, fp64 sum rounded
once to fp32) against facts that do not come from the oracle itself."""

import math

import numpy as np
import pytest

from oracle import moe_oracle as o


def _bf16_bits(v):
    return o.f64_to_bf16_bits(o.bf16_round(np.asarray(v, dtype=np.float64)))


def test_one_hot_rows_select_gate_columns():
    """x = unit vector e_h picks column h of every gate row: logits[t, e] = W_g[e, h(t)].
    A transposed or mis-indexed product fails this (E != H)."""
    rng = np.random.default_rng(0)
    E, H, T = 5, 16, 16
    wg = rng.standard_normal((E, H)).astype(np.float32)
    x = np.eye(T, H)
    lg = o.router_logits(_bf16_bits(x), wg)
    assert lg.shape == (T, E)
    np.testing.assert_array_equal(lg, wg.T[:T].astype(np.float64))


def test_integer_inputs_exact():
    """Small-integer x (exact in bf16) and W_g: the dot products are exact integers,
    checked against Python integer arithmetic."""
    rng = np.random.default_rng(1)
    T, H, E = 6, 48, 7
    xi = rng.integers(-8, 9, size=(T, H))
    wi = rng.integers(-100, 101, size=(E, H))
    lg = o.router_logits(_bf16_bits(xi), wi.astype(np.float32))
    for t in range(T):
        for e in range(E):
            assert lg[t, e] == sum(int(xi[t, h]) * int(wi[e, h]) for h in range(H))


def test_matches_correctly_rounded_sum():
    """Random inputs: each logit equals the correctly rounded fp32 value of the exact
    dot product (math.fsum over exact fp64 products of bf16 x fp32 values), up to one
    fp32 ulp for the rare double-rounding case."""
    rng = np.random.default_rng(2)
    T, H, E = 4, 256, 9
    xb = _bf16_bits(rng.standard_normal((T, H)))
    wg = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    lg = o.router_logits(xb, wg)
    assert np.all(lg.astype(np.float32).astype(np.float64) == lg), "not fp32 values"
    xv = o.bf16_bits_to_f64(xb)
    for t in range(T):
        for e in range(E):
            exact = math.fsum(float(xv[t, h]) * float(wg[e, h]) for h in range(H))
            ref = float(np.float32(exact))
            assert abs(lg[t, e] - ref) <= abs(ref) * 2.0 ** -23 + 1e-30


def test_routing_on_projected_logits_is_the_gate_argmax():
    """k = 1 routing of the projected logits picks argmax_e of x . W_g[e] (brute force)."""
    rng = np.random.default_rng(3)
    T, H, E = 10, 64, 12
    xb = _bf16_bits(rng.standard_normal((T, H)))
    wg = rng.standard_normal((E, H)).astype(np.float32)
    lg = o.router_logits(xb, wg)
    idx, w = o.route(lg, 1)
    xv = o.bf16_bits_to_f64(xb)
    for t in range(T):
        scores = [math.fsum(xv[t] * wg[e].astype(np.float64)) for e in range(E)]
        assert idx[t, 0] == int(np.argmax(scores))
        assert w[t, 0] == pytest.approx(1.0)
