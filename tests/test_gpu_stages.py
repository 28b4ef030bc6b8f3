"""GPU parity of each stage against the oracle, through the C interface.

Bit-exact: routing indices, histogram, offsets, permutation, inverse map, FP8 codes
and scales of the activation quantisation, and the grouped GEMMs on exact-integer
inputs.  Floating point: max|err| <= 2e-2 * RMS(ref), cosine >= 0.9999."""

import numpy as np
import pytest
import torch

import moe_expert_ffn_scan_gb300 as moe
from gen import inputs as gi
from oracle import moe_oracle as o
from tests._parity import (assert_float_close, assert_fp8_codes_close, bf16_np, bits_np)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _status_ok(ws):
    bits = moe.moe_check_status(ws)
    assert bits == 0, f"device status bits {bits:#x}"


# ------------------------------------------------------------------ a3 quant ---------

@pytest.mark.parametrize("rows,cols", [(64, 512), (7, 7168), (1, 128), (333, 1024)])
def test_quant_act_bit_exact(rows, cols):
    x = gi.activations(rows, cols, seed=rows, device="cpu")
    # special blocks: zeros, negative zeros, a block whose amax is exactly 448*2^e,
    # one just above it, tiny and huge magnitudes
    x[0, :128] = 0.0
    if rows > 1:
        x[1, :128] = -0.0
    if rows > 2:
        x[2, :128] = torch.linspace(-3.5, 3.5, 128).to(torch.bfloat16)  # amax 3.5 = 448*2^-7
    if rows > 3:
        x[3, :128] = x[3, :128] * 1e-30
    if rows > 4:
        x[4, :128] = x[4, :128] * 1e30
    xg = x.to(DEV)
    q = torch.empty(rows, cols, dtype=torch.uint8, device=DEV)
    s = torch.empty(rows, cols // 128, dtype=torch.uint8, device=DEV)
    moe.moe_quant_act(xg, q, s)
    torch.cuda.synchronize()
    rq, rs = o.quant_act(bits_np(x))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


# ------------------------------------------------------------------ a1 + a2 route ----

def _run_route(d, logits):
    T, E, k, sh = d.T, d.E, d.k, d.has_shared
    R = T * k
    G = E + sh
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(G + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(R, dtype=torch.int32, device=DEV)
    inv = torch.empty(R, dtype=torch.int32, device=DEV)
    ws = moe.alloc_workspace(moe.route_workspace_size(d))
    moe.moe_route(d, logits.to(DEV), idx, w, counts, offsets, perm, inv, ws)
    _status_ok(ws)
    return [t.cpu().numpy() for t in (idx, w, counts, offsets, perm, inv)]


@pytest.mark.parametrize("T,E,k,sh,kind", [(64, 8, 2, 0, "normal"), (7, 384, 8, 1, "normal"),
                                           (256, 384, 8, 1, "zipf"), (1000, 384, 8, 1, "zipf"),
                                           (300, 1024, 16, 1, "normal"), (5, 3, 3, 0, "normal"),
                                           (1, 33, 1, 1, "normal"), (600, 20, 4, 0, "normal")])
def test_route_bit_exact(T, E, k, sh, kind):
    d = moe.dims(T, 128, 128, E, k, sh)
    if kind == "zipf":
        lg = gi.zipf_logits(T, E, seed=T, device="cpu")
    else:
        lg = torch.randn(T, E, generator=torch.Generator().manual_seed(T * E))
    idx, w, counts, offsets, perm, inv = _run_route(d, lg)
    ridx, rw = o.route(lg.numpy(), k)
    rc, roff, rperm, rinv = o.permute(ridx, E, sh)
    assert np.array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-7)
    assert np.array_equal(counts, rc)
    assert np.array_equal(offsets, roff)
    assert np.array_equal(perm, rperm)
    assert np.array_equal(inv, rinv)


def test_route_ties_and_duplicates():
    T, E, k = 40, 16, 4
    lg = torch.randint(0, 3, (T, E)).float()  # many exact ties
    d = moe.dims(T, 128, 128, E, k, 0)
    idx, w, counts, offsets, perm, inv = _run_route(d, lg)
    ridx, rw = o.route(lg.numpy(), k)
    assert np.array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=2e-6)
    rc, roff, rperm, rinv = o.permute(ridx, E, 0)
    assert np.array_equal(perm, rperm) and np.array_equal(inv, rinv)


# ------------------------------------------------------------------ a4/a6 GEMM -------

def _gemm_case(G, N, K, sizes, seed, integer):
    rows = int(sum(sizes))
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    if integer:
        aq = gi.integer_codes((rows, K), gi.E4M3_INTEGER_CODES, seed, "cpu", "act")
        asc = torch.full((rows, K // 128), 127, dtype=torch.uint8)
        wq = gi.integer_fp4_bytes((G, N, K // 2), seed, "cpu", "w13")
        wsc = torch.full((G, N, K // 32), 127, dtype=torch.uint8)
    else:
        x = gi.activations(rows, K, seed, "cpu", name="act")
        q, s = o.quant_act(bits_np(x))
        aq, asc = torch.from_numpy(q), torch.from_numpy(s)
        wq, wsc = gi.mxfp4_weights(G, N, K, seed, "cpu")
    return offsets, aq, asc, wq, wsc


def _run_gemm(which, G, N, K, offsets, aq, asc, wq, wsc):
    rows = int(offsets[-1])
    # express the call as a layer with `rows` packed rows, one route per token
    if which == "w13":
        d = moe.dims(max(rows, 1), K, N // 2, G, 1, 0)
    else:
        d = moe.dims(max(rows, 1), N, K, G, 1, 0)
    y = torch.full((max(rows, 1), N), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(moe.gemm_workspace_size(d))
    off = torch.from_numpy(offsets).to(DEV)
    if which == "w13":
        moe.moe_grouped_gemm_w13(d, aq.to(DEV), asc.to(DEV), None, off, wq.to(DEV),
                                 wsc.to(DEV), y, ws)
    else:
        moe.moe_grouped_gemm_w2(d, aq.to(DEV), asc.to(DEV), off, wq.to(DEV), wsc.to(DEV), y, ws)
    _status_ok(ws)
    return bf16_np(y[:rows])


GEMM_SHAPES = [
    ("w13", 3, 256, 512, [5, 0, 11]),
    ("w2", 2, 512, 256, [1, 2]),
    ("w13", 4, 512, 1024, [16, 17, 33, 130]),
    ("w2", 3, 256, 384, [300, 7, 128]),
    ("w13", 2, 256, 128, [1, 64]),
    ("w2", 3, 1024, 3072, [1, 40, 200]),
    ("w13", 5, 512, 512, [0, 16, 64, 65, 129]),
    ("w13", 2, 256, 512, [224, 150]),
    # more small-group tiles than one wave of CTAs: full waves, then a split last wave
    ("w13", 40, 1024, 640, [(i * 7) % 17 for i in range(40)]),
    ("w2", 24, 2048, 1536, [(i * 5) % 16 + 1 for i in range(24)]),
    # decode-like: long K (28 two-sub-tile stages), 1-7 rows per group
    ("w13", 6, 1024, 7168, [1, 2, 7, 1, 0, 3]),
    # the medium tiles' lower range (17..33 rows, around the 32-row mark), many tiles,
    # long and odd K
    ("w13", 6, 1024, 1024, [17, 32, 16, 33, 24, 31]),
    ("w2", 4, 512, 3072, [20, 32, 17, 29]),
    ("w13", 3, 256, 640, [18, 25, 32]),
    ("w13", 2, 512, 7168, [32, 21]),
    # mid variant: one chunk of 65..128 rows, or two of <= 128 (M = 241..256)
    ("w13", 3, 512, 1024, [256, 100, 250]),
    ("w2", 2, 1024, 640, [80, 128]),        # K/128 odd: one-sub-tile stages
    # large variant: many weight tiles, long K with quads of scale bytes in flight, and
    # N not a multiple of 256
    ("w2", 2, 1536, 1536, [200, 129]),
    ("w13", 3, 512, 7168, [224, 0, 190]),
    ("w2", 2, 384, 512, [200, 150]),
]


@pytest.mark.parametrize("which,G,N,K,sizes", GEMM_SHAPES)
def test_grouped_gemm_exact_integer(which, G, N, K, sizes):
    offsets, aq, asc, wq, wsc = _gemm_case(G, N, K, sizes, seed=G * N + K, integer=True)
    y = _run_gemm(which, G, N, K, offsets, aq, asc, wq, wsc)
    ref = o.grouped_gemm(aq.numpy(), asc.numpy(), offsets, wq.numpy(), wsc.numpy())
    bad = np.argwhere(y != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}: " \
                          f"got {y[tuple(bad[0])]} want {ref[tuple(bad[0])]}"


@pytest.mark.parametrize("which,G,N,K,sizes", GEMM_SHAPES)
def test_grouped_gemm_random_mxfp4(which, G, N, K, sizes):
    offsets, aq, asc, wq, wsc = _gemm_case(G, N, K, sizes, seed=G + N + K, integer=False)
    y = _run_gemm(which, G, N, K, offsets, aq, asc, wq, wsc)
    ref = o.grouped_gemm(aq.numpy(), asc.numpy(), offsets, wq.numpy(), wsc.numpy())
    assert_float_close(y, ref, f"{which} y")


@pytest.mark.parametrize("sizes", [[3, 20], [3, 200]])
def test_grouped_gemm_scale_addressing(sizes):
    """Non-unit weight scales at one (row, 32-block) and activation scale at one
    (row, 128-block): bit-exact on integer inputs (small variant; large variant, with
    weight rows 129 and 200 in the second 128-row tile and token 150 in the second
    token-scale atom)."""
    G, N, K = 2, 256, 512
    offsets, aq, asc, wq, wsc = _gemm_case(G, N, K, sizes, seed=99, integer=True)
    wsc = wsc.clone()
    asc = asc.clone()
    wsc[1, 200, 5] = 128
    wsc[0, 3, 15] = 125
    wsc[1, 129, 0] = 126
    asc[10, 2] = 128
    asc[1, 0] = 125
    if offsets[-1] > 150:
        asc[150, 3] = 126  # a token past the first 128 of a large-variant chunk
    y = _run_gemm("w13", G, N, K, offsets, aq, asc, wq, wsc)
    ref = o.grouped_gemm(aq.numpy(), asc.numpy(), offsets, wq.numpy(), wsc.numpy())
    assert np.array_equal(y, ref)


# ------------------------------------------------------------------ a5 swiglu+quant --

@pytest.mark.parametrize("rows,I", [(128, 256), (63, 3072), (1, 128)])
def test_swiglu_quant(rows, I):
    rng = np.random.default_rng(rows + I)
    y13 = o.bf16_round(rng.standard_normal((rows, 2 * I)) * 40.0)
    y13_t = torch.from_numpy(y13).to(torch.bfloat16)
    hq = torch.empty(rows, I, dtype=torch.uint8, device=DEV)
    hs = torch.empty(rows, I // 128, dtype=torch.uint8, device=DEV)
    moe.moe_swiglu_quant(y13_t.to(DEV), hq, hs)
    torch.cuda.synchronize()
    rq, rs = o.swiglu_quant(y13)
    rate = assert_fp8_codes_close(hq.cpu().numpy(), hs.cpu().numpy(), rq, rs, "hq",
                                  max_mismatch=1e-3)
    assert rate > 0.999


# ------------------------------------------------------------------ a7 combine -------

@pytest.mark.parametrize("T,H,k,sh", [(64, 512, 2, 0), (7, 7168, 8, 1), (33, 256, 3, 1)])
def test_combine(T, H, k, sh):
    rng = np.random.default_rng(T * k)
    R = T * k
    Rs = R + (T if sh else 0)
    y2 = o.bf16_round(rng.standard_normal((Rs, H)) * 100)
    inv = rng.permutation(R).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    d = moe.dims(T, H, 128, max(k, 8), k, sh)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(d, torch.from_numpy(y2).to(torch.bfloat16).to(DEV),
                    torch.from_numpy(inv).to(DEV), torch.from_numpy(w).to(DEV), out)
    torch.cuda.synchronize()
    ref = o.combine(y2, inv, w.astype(np.float64), T, k, sh)
    assert_float_close(bf16_np(out), ref, "out")
    # fp32 sums of k <= 8 bf16 terms round to the same bf16 in almost every element
    assert np.mean(bf16_np(out) != ref) < 1e-2


@pytest.mark.parametrize("K", [512, 384])
@pytest.mark.parametrize("M", [224, 240])
def test_grouped_gemm_token_scales_beyond_128_rows(K, M):
    """One large-variant chunk of M token rows (two token-scale atoms): every row gets
    its own activation scale byte, integer codes keep the result exact."""
    G, N = 1, 256
    sizes = [M]
    offsets, aq, asc, wq, wsc = _gemm_case(G, N, K, sizes, seed=7, integer=True)
    asc = (125 + (torch.arange(M).view(M, 1) * 7 + torch.arange(K // 128).view(1, -1)) % 5
           ).to(torch.uint8)
    wsc = (124 + torch.randint(0, 5, wsc.shape, generator=torch.Generator().manual_seed(3))
           ).to(torch.uint8)
    y = _run_gemm("w13", G, N, K, offsets, aq, asc, wq, wsc)
    ref = o.grouped_gemm(aq.numpy(), asc.numpy(), offsets, wq.numpy(), wsc.numpy())
    bad = np.argwhere(y != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, rows {np.unique(bad[:, 0])[:10]}"
