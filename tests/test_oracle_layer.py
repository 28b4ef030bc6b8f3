"""Pins for the oracle's routing, permutation, grouped GEMM, SwiGLU and combine
(CPU only).  Independent checks: brute-force selection loops, library softmax,
closed-form GEMM results on structured inputs, invariants, and a dense unrouted
recomputation of the whole layer."""

import numpy as np
import pytest
import scipy.special
import torch

from gen import inputs as gi
from oracle import moe_oracle as o
from tests._parity import with_gate_logits


def _tiny():
    d, t = gi.make_layer("tiny")
    return d, with_gate_logits(t)


def _bits(x_bf16):
    return x_bf16.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- route -------------

def _brute_topk(row, k):
    taken = []
    for _ in range(k):
        best = None
        for e in range(len(row)):
            if e not in taken and (best is None or row[e] > row[best]):
                best = e
        taken.append(best)
    return taken


@pytest.mark.parametrize("T,E,k", [(50, 8, 2), (20, 384, 8), (9, 33, 5), (4, 16, 16), (3, 7, 1)])
def test_route_matches_brute_force_and_softmax(T, E, k):
    rng = np.random.default_rng(T * E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = o.route(lg, k)
    for t in range(T):
        assert list(idx[t]) == _brute_topk(lg[t].astype(np.float64), k)
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0) and np.all(w > 0) and np.all(w <= 1)


def test_route_ties_lower_index_first():
    lg = np.array([[1.0, 3.0, 3.0, 0.5, 3.0, -1.0],
                   [2.0, 2.0, 2.0, 2.0, 2.0, 2.0]], dtype=np.float32)
    idx, w = o.route(lg, 3)
    assert idx.tolist() == [[1, 2, 4], [0, 1, 2]]
    np.testing.assert_allclose(w, 1.0 / 3.0, rtol=1e-15)


# ---------------------------------------------------------------- permute -----------

def _counting_sort_permute(idx, E, has_shared):
    """Independent loop version: walk experts, then tokens in order."""
    T, k = len(idx), len(idx[0])
    perm = []
    counts = [0] * E
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t][j] == e:
                    perm.append(t * k + j)
                    counts[e] += 1
    offs = [0]
    for c in counts + ([T] if has_shared else []):
        offs.append(offs[-1] + c)
    return counts, offs, perm


@pytest.mark.parametrize("T,E,k,sh", [(64, 8, 2, 0), (7, 384, 8, 1), (33, 40, 8, 1), (1, 4, 4, 0)])
def test_permute_invariants_and_counting_sort(T, E, k, sh):
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = o.route(lg, k)
    counts, offsets, perm, inv = o.permute(idx, E, sh)
    c2, off2, perm2 = _counting_sort_permute(idx.tolist(), E, sh)
    assert counts.tolist() == c2 and offsets.tolist() == off2 and perm.tolist() == perm2
    R = T * k
    assert counts.sum() == R and offsets[E] == R and offsets[-1] == R + (T if sh else 0)
    assert sorted(perm.tolist()) == list(range(R))
    assert np.array_equal(inv[perm], np.arange(R))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(idx.reshape(-1)[seg] == e)
        assert np.all(np.diff(seg // k) > 0)
    # each token has exactly k distinct experts
    assert all(len(set(r)) == k for r in idx.tolist())


# ---------------------------------------------------------------- grouped GEMM ------

def _int_act(rows, K, seed):
    codes = gi.integer_codes((rows, K), gi.E4M3_INTEGER_CODES, seed, "cpu", "act").numpy()
    return codes, np.full((rows, K // 128), 127, np.uint8)


def _fp4_from_vals(vals):
    """float values in the E2M1 integer set -> packed code bytes (test helper)."""
    lut = {0.0: 0x0, 1.0: 0x2, 2.0: 0x4, 3.0: 0x5, 4.0: 0x6, 6.0: 0x7,
           -1.0: 0xA, -2.0: 0xC, -3.0: 0xD, -4.0: 0xE, -6.0: 0xF}
    c = np.vectorize(lambda v: lut[float(v)])(vals).astype(np.uint8)
    return c[..., 0::2] | (c[..., 1::2] << 4)


def test_grouped_gemm_selection_matrices():
    """W[g][n][k] = 1 iff k == sigma_g(n): y[r, n] must be x[r, sigma_g(n)] exactly.
    Pins operand orientation, nibble order and group indexing."""
    rng = np.random.default_rng(5)
    G, N, K = 3, 40, 256
    sizes = [5, 0, 11]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    aq, asc = _int_act(offsets[-1], K, 6)
    xv = o.e4m3_decode(aq)
    W = np.zeros((G, N, K))
    sig = [rng.permutation(K)[:N] for _ in range(G)]
    for g in range(G):
        W[g, np.arange(N), sig[g]] = 1.0
    wq = _fp4_from_vals(W)
    ws = np.full((G, N, K // 32), 127, np.uint8)
    y = o.grouped_gemm(aq, asc, offsets, wq, ws)
    for g in range(G):
        for r in range(offsets[g], offsets[g + 1]):
            assert np.array_equal(y[r], xv[r, sig[g]])


def test_grouped_gemm_exact_integer_dot_products():
    rng = np.random.default_rng(7)
    G, N, K = 2, 24, 512
    offsets = np.array([0, 6, 13], np.int32)
    aq, asc = _int_act(13, K, 8)
    vals = rng.choice([0, 1, 2, 3, 4, 6, -1, -2, -3, -4, -6], size=(G, N, K)).astype(np.float64)
    wq = _fp4_from_vals(vals)
    ws = np.full((G, N, K // 32), 127, np.uint8)
    y = o.grouped_gemm(aq, asc, offsets, wq, ws)
    xv = o.e4m3_decode(aq)
    for g in range(G):
        for r in range(offsets[g], offsets[g + 1]):
            for n in range(N):
                exact = int(sum(int(a) * int(b) for a, b in zip(xv[r], vals[g, n])))
                assert y[r, n] == float(o.bf16_round(np.float64(exact)))


def test_grouped_gemm_scale_addressing():
    """One weight scale byte (row n0, K-block b0) and one activation scale byte
    (row r0, 128-block c0) set to 128 (x2): exactly those contributions double."""
    G, N, K = 1, 8, 256
    offsets = np.array([0, 4], np.int32)
    aq, asc = _int_act(4, K, 9)
    xv = o.e4m3_decode(aq)
    ones = np.ones((G, N, K))
    wq = _fp4_from_vals(ones)
    ws = np.full((G, N, K // 32), 127, np.uint8)
    n0, b0, r0, c0 = 5, 3, 2, 1
    ws[0, n0, b0] = 128
    asc = asc.copy()
    asc[r0, c0] = 128
    y = o.grouped_gemm(aq, asc, offsets, wq, ws)
    for r in range(4):
        a = xv[r].copy()
        if r == r0:
            a[c0 * 128:(c0 + 1) * 128] *= 2
        for n in range(N):
            wrow = np.ones(K)
            if n == n0:
                wrow[b0 * 32:(b0 + 1) * 32] = 2
            assert y[r, n] == o.bf16_round(np.float64(np.dot(a, wrow)))


# ---------------------------------------------------------------- swiglu / combine --

def test_swiglu_closed_forms():
    g = np.array([[0.0, 1.0, -2.0, 30.0, -30.0, 0.5]])
    u = np.array([[5.0, 2.0, 3.0, 1.0, 7.0, -4.0]])
    h = o.swiglu(np.concatenate([g, u], axis=1))
    want = g * scipy.special.expit(g) * u
    np.testing.assert_allclose(h, want, rtol=1e-14, atol=1e-300)
    assert h[0, 0] == 0.0


def test_swiglu_quant_uses_fp32_h():
    rng = np.random.default_rng(11)
    y13 = o.bf16_round(rng.standard_normal((6, 512)) * 30)
    hq, hs = o.swiglu_quant(y13)
    q2, s2 = o.quant_rows(o.swiglu(y13).astype(np.float32).astype(np.float64))
    assert np.array_equal(hq, q2) and np.array_equal(hs, s2)
    assert hq.shape == (6, 256) and hs.shape == (6, 2)


def test_combine_k1_identity_and_shared_add():
    rng = np.random.default_rng(12)
    T, H = 5, 64
    y2 = o.bf16_round(rng.standard_normal((2 * T, H)))
    inv = np.array([3, 0, 4, 1, 2])
    out = o.combine(y2, inv, np.ones((T, 1)), T, 1, 0)
    assert np.array_equal(out, y2[inv])
    out2 = o.combine(y2, inv, np.ones((T, 1)), T, 1, 1)
    assert np.array_equal(out2, o.bf16_round(y2[inv] + y2[T:]))


# ---------------------------------------------------------------- whole layer -------

def _np_layer(t):
    return (_bits(t["x"]), t["logits"].numpy(), t["w13"].numpy(), t["w13_s"].numpy(),
            t["w2"].numpy(), t["w2_s"].numpy())


def test_dense_unrouted_equals_routed_tiny():
    d, t = _tiny()
    x, lg, w13, w13s, w2, w2s = _np_layer(t)
    r = o.moe_forward(x, lg, d.k, w13, w13s, w2, w2s, d.has_shared)
    dense = o.dense_unrouted_forward(x, lg, d.k, w13, w13s, w2, w2s, d.has_shared)
    assert np.array_equal(r["out"], dense)
    assert r["counts"].sum() == d.T * d.k


def test_dense_unrouted_equals_routed_with_shared_ragged():
    d = gi.Dims(T=13, H=256, I=128, E=5, k=3, has_shared=1)
    t = gi.custom_layer(d, seed=3)
    x, lg, w13, w13s, w2, w2s = _np_layer(t)
    r = o.moe_forward(x, lg, d.k, w13, w13s, w2, w2s, d.has_shared)
    dense = o.dense_unrouted_forward(x, lg, d.k, w13, w13s, w2, w2s, d.has_shared)
    assert np.array_equal(r["out"], dense)
    assert r["offsets"][-1] == d.Rs


def test_zero_input_gives_zero_output():
    d, t = _tiny()
    t["x"] = torch.zeros_like(t["x"])
    x, lg, w13, w13s, w2, w2s = _np_layer(t)
    r = o.moe_forward(x, lg, d.k, w13, w13s, w2, w2s, d.has_shared)
    assert np.all(r["out"] == 0) and np.all(r["xs"] == 127) and np.all(r["hs"] == 127)


def test_token_subset_matches_full_layer():
    d, t = _tiny()
    x, lg, w13, w13s, w2, w2s = _np_layer(t)
    full = o.moe_forward(x, lg, d.k, w13, w13s, w2, w2s, d.has_shared)
    sub = o.moe_forward_tokens(x, lg, d.k, w13, w13s, w2, w2s, d.has_shared, [3, 17, 60])
    assert np.array_equal(sub["out"], full["out"][[3, 17, 60]])
