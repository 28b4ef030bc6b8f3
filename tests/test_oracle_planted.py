"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of an oracle function -- a wrong sign, bias,
rounding, tie rule, index order, block size, operand order or dropped term -- swaps
it into the oracle module for the duration of the case, and runs the pin that should
notice it; the pin must fail.  The mistakes live here, in the oracle, on the CPU:
nothing touches the CUDA path.
"""

import numpy as np
import pytest

from oracle import moe_oracle as o
from tests import test_oracle_formats as tf
from tests import test_oracle_layer as tl
from tests import test_oracle_nvfp4 as tn
from tests import test_oracle_router as tr


# ------------------------------------------------------------ the planted mistakes --

def _e2m1_no_sign(codes):
    return np.abs(_orig["e2m1_decode"](codes))


def _e2m1_bias0(codes):  # exponent bias 0 instead of 1
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    exp, man = (c >> 1) & 0x3, c & 0x1
    return sign * np.where(exp == 0, 0.5 * man, np.ldexp(1.0 + 0.5 * man, exp))


def _e8m0_bias128(b):
    return _orig["e8m0_decode"](b) * 0.5


def _e4m3_ties_away(v):  # round half away from zero instead of to the even code
    v = np.asarray(v, dtype=np.float64)
    pos = o._E4M3_POS
    a = np.minimum(np.abs(v), o.E4M3_MAX)
    hi = np.minimum(np.searchsorted(pos, a, side="left"), 0x7E)
    lo = np.maximum(hi - 1, 0)
    pick_hi = (pos[hi] - a) <= (a - pos[lo])
    code = np.where(pos[hi] == a, hi, np.where(pick_hi, hi, lo))
    return (code | np.where(np.signbit(v), 0x80, 0x00)).astype(np.uint8)


def _scale_exp_plus1(amax):
    return _orig["scale_exponent"](amax) + 1


def _scale_exp_strict(amax):  # amax == 448 * 2**e pushed one exponent up
    amax = np.asarray(amax, dtype=np.float64)
    f, p = np.frexp(amax)
    e = np.where(f < 0.875, p - 9, p - 8)
    return np.clip(np.where(amax == 0, 0, e), -127, 127).astype(np.int64)


def _bf16_truncate(v):
    v = np.asarray(v, dtype=np.float64)
    _, p = np.frexp(v)
    ulp = np.ldexp(1.0, np.maximum(p - 8, -133))
    return np.trunc(v / ulp) * ulp


def _mxfp4_high_nibble_first(codes, scales):
    codes = np.asarray(codes)
    swapped = ((codes & 0xF) << 4) | (codes >> 4)
    return _orig["mxfp4_dequant"](swapped.astype(np.uint8), scales)


def _mxfp4_block16(codes, scales):  # scale byte indexed by K // 16 instead of K // 32
    codes = np.asarray(codes)
    n, kh = codes.shape
    k = kh * 2
    vals = np.empty((n, k))
    vals[:, 0::2] = o.e2m1_decode(codes & 0xF)
    vals[:, 1::2] = o.e2m1_decode(codes >> 4)
    s = o.e8m0_decode(scales)
    s16 = s[:, np.minimum(np.arange(k // 16), s.shape[1] - 1)]
    return (vals.reshape(n, k // 16, 16) * s16[:, :, None]).reshape(n, k)


def _nvfp4_block32(codes, scales, global_scale=None):  # one E4M3 scale per 32 K
    codes = np.asarray(codes)
    n, kh = codes.shape
    k = kh * 2
    vals = np.empty((n, k))
    vals[:, 0::2] = o.e2m1_decode(codes & 0xF)
    vals[:, 1::2] = o.e2m1_decode(codes >> 4)
    s = o.e4m3_decode(scales)[:, :k // 32]
    w = (vals.reshape(n, k // 32, 32) * s[:, :, None]).reshape(n, k)
    if global_scale is not None:
        gs = np.atleast_1d(np.asarray(global_scale, dtype=np.float32).astype(np.float64))
        w = w * np.repeat(gs, n // len(gs))[:, None]
    return w


def _nvfp4_one_tensor_scale(codes, scales, global_scale=None):  # gate scale on every row
    if global_scale is not None:
        global_scale = np.atleast_1d(np.asarray(global_scale, dtype=np.float32))[:1]
    return _orig["nvfp4_dequant"](codes, scales, global_scale)


def _quant_rows_block64(x):  # one scale per 64 columns instead of 128
    x = np.asarray(x, dtype=np.float64)
    rows, cols = x.shape
    xb = x.reshape(rows, cols // 64, 64)
    e = o.scale_exponent(np.abs(xb).max(axis=2))
    codes = o.e4m3_encode(np.ldexp(xb, -e[:, :, None]))
    return codes.reshape(rows, cols), (e + 127).astype(np.uint8)


def _router_fp32_running_sum(x_bf16_bits, wg):  # fp32 accumulation, term by term
    x = o.bf16_bits_to_f64(x_bf16_bits).astype(np.float32)
    w = np.asarray(wg, dtype=np.float32)
    acc = np.zeros((x.shape[0], w.shape[0]), np.float32)
    for h in range(x.shape[1]):
        acc = acc + x[:, h:h + 1] * w[None, :, h]
    return acc.astype(np.float64)


def _route_ties_high(logits, k):  # equal logits -> higher expert index first
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = lg.shape
    order = np.lexsort((-np.broadcast_to(np.arange(E), (T, E)), -lg), axis=-1)
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(lg, idx.astype(np.int64), axis=1)
    ex = np.exp(sel - sel[:, :1])
    return idx, ex / ex.sum(axis=1, keepdims=True)


def _route_full_softmax(logits, k):  # weights not renormalised over the selected k
    idx, _ = _orig["route"](logits, k)
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return idx, np.take_along_axis(p, idx.astype(np.int64), axis=1)


def _permute_tokens_descending(idx, E, has_shared):
    counts, offsets, perm, _ = _orig["permute"](idx, E, has_shared)
    perm = perm.copy()
    for e in range(E):
        perm[offsets[e]:offsets[e + 1]] = perm[offsets[e]:offsets[e + 1]][::-1]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    return counts, offsets, perm, inv


def _swiglu_swapped(y13):  # silu(up) * gate
    y13 = np.asarray(y13, dtype=np.float64)
    I = y13.shape[1] // 2
    u, g = y13[:, :I], y13[:, I:]
    return g / (1.0 + np.exp(-g)) * u


def _combine_no_shared(y2, inv, w, T, k, has_shared):
    return _orig["combine"](y2, inv, w, T, k, 0)


def _combine_inv_transposed(y2, inv, w, T, k, has_shared):  # inv read as [k, T]
    inv_t = np.asarray(inv).reshape(k, T).T.reshape(-1) if k > 1 else np.asarray(inv)
    return _orig["combine"](y2, inv_t, w, T, k, has_shared)


_orig = {n: getattr(o, n) for n in (
    "e2m1_decode", "e8m0_decode", "scale_exponent", "mxfp4_dequant", "nvfp4_dequant",
    "route", "permute", "combine")}


CASES = [
    ("E2M1 sign bit ignored", "e2m1_decode", _e2m1_no_sign,
     tf.test_e2m1_matches_spec_table),
    ("E2M1 exponent bias 0", "e2m1_decode", _e2m1_bias0, tf.test_e2m1_times_e8m0_exhaustive),
    ("E8M0 bias 128", "e8m0_decode", _e8m0_bias128, tf.test_e8m0_matches_spec_and_torch),
    ("E4M3 ties away from zero", "e4m3_encode", _e4m3_ties_away,
     tf.test_e4m3_encode_midpoints_ties_to_even),
    ("scale exponent one too large", "scale_exponent", _scale_exp_plus1,
     tf.test_scale_exponent_brute_force_minimal),
    ("scale exponent boundary excluded", "scale_exponent", _scale_exp_strict,
     tf.test_scale_exponent_landmarks),
    ("bf16 truncated instead of rounded", "bf16_round", _bf16_truncate,
     tf.test_bf16_round_float64_is_nearest_ties_even),
    ("MXFP4 high nibble = even K", "mxfp4_dequant", _mxfp4_high_nibble_first,
     tl.test_grouped_gemm_selection_matrices),
    ("MXFP4 scale per 16 K", "mxfp4_dequant", _mxfp4_block16,
     tl.test_grouped_gemm_scale_addressing),
    ("NVFP4 scale per 32 K", "nvfp4_dequant", _nvfp4_block32,
     tn.test_nvfp4_scale_block_is_16_elements),
    ("NVFP4 one tensor scale for gate and up", "nvfp4_dequant", _nvfp4_one_tensor_scale,
     tn.test_nvfp4_tensor_scale_per_row_segment),
    ("FP8 activation block of 64", "quant_rows", _quant_rows_block64,
     tf.test_quant_rows_properties),
    ("router logits summed in fp32", "router_logits", _router_fp32_running_sum,
     tr.test_matches_correctly_rounded_sum),
    ("top-k ties to the higher index", "route", _route_ties_high,
     tl.test_route_ties_lower_index_first),
    ("top-k weights not renormalised", "route", _route_full_softmax,
     lambda: tl.test_route_matches_brute_force_and_softmax(50, 8, 2)),
    ("tokens descending inside a group", "permute", _permute_tokens_descending,
     lambda: tl.test_permute_invariants_and_counting_sort(64, 8, 2, 0)),
    ("gate and up swapped", "swiglu", _swiglu_swapped, tl.test_swiglu_closed_forms),
    ("shared-expert row dropped", "combine", _combine_no_shared,
     tl.test_combine_k1_identity_and_shared_add),
    ("inverse map read transposed", "combine", _combine_inv_transposed,
     tl.test_dense_unrouted_equals_routed_with_shared_ragged),
]


@pytest.mark.parametrize("name,func,mutant,pin", CASES, ids=[c[0] for c in CASES])
def test_pin_catches_planted_mistake(monkeypatch, name, func, mutant, pin):
    monkeypatch.setattr(o, func, mutant)
    with pytest.raises(AssertionError):
        pin()


@pytest.mark.parametrize("name,func,mutant,pin", CASES, ids=[c[0] for c in CASES])
def test_pin_passes_on_the_oracle(name, func, mutant, pin):
    """The same pins pass on the unmodified oracle (so a failure above is the
    planted mistake's)."""
    pin()
