"""GPU parity of the NVFP4-weight path (f3; GB10 "Optimization progress report",
Optimization 05) against the oracle, through the C interface: the grouped GEMMs
bit-exact on exact-integer inputs across every tile variant, within the float
tolerance on random NVFP4 weights, and whole layers (tiny, ragged, full-size decode)."""

import numpy as np
import pytest
import torch

import moe_expert_ffn_scan_gb300 as moe
from gen import inputs as gi
from oracle import moe_oracle as o
from tests._parity import (assert_float_close, assert_fp8_codes_close, bf16_np, bits_np,
                           with_gate_logits)

pytestmark = pytest.mark.gpu

DEV = "cuda"

# E4M3 block scales 1, 2, 3 (integer products stay exact) and power-of-two tensor scales
INT_SCALES = (0x38, 0x40, 0x44)


def _nv_case(which, G, N, K, sizes, seed, integer):
    rows = int(sum(sizes))
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    S = 2 if which == "w13" else 1
    if integer:
        aq = gi.integer_codes((rows, K), gi.E4M3_INTEGER_CODES, seed, "cpu", "act")
        asc = torch.full((rows, K // 128), 127, dtype=torch.uint8)
        wq = gi.integer_fp4_bytes((G, N, K // 2), seed, "cpu", "w13")
        wsc = gi.integer_codes((G, N, K // 16), INT_SCALES, seed, "cpu", "w13_s")
        gs = torch.tensor([0.5, 1.0, 2.0])[torch.randint(
            0, 3, (G, S), generator=torch.Generator().manual_seed(seed))]
    else:
        x = gi.activations(rows, K, seed, "cpu", name="act")
        q, s = o.quant_act(bits_np(x))
        aq, asc = torch.from_numpy(q), torch.from_numpy(s)
        wq, wsc, gs = gi.nvfp4_weights(G, N, K, seed, "cpu", segments=S)
    return offsets, aq, asc, wq, wsc, gs.to(torch.float32).contiguous()


def _run_nv(which, G, N, K, offsets, aq, asc, wq, wsc, gs):
    rows = int(offsets[-1])
    if which == "w13":
        d = moe.dims(max(rows, 1), K, N // 2, G, 1, 0)
    else:
        d = moe.dims(max(rows, 1), N, K, G, 1, 0)
    y = torch.full((max(rows, 1), N), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(moe.gemm_workspace_size_nvfp4(d))
    off = torch.from_numpy(offsets).to(DEV)
    g = gs.to(DEV)
    if which == "w13":
        moe.moe_grouped_gemm_w13_nvfp4(d, aq.to(DEV), asc.to(DEV), None, off, wq.to(DEV),
                                       wsc.to(DEV), g, y, ws)
    else:
        moe.moe_grouped_gemm_w2_nvfp4(d, aq.to(DEV), asc.to(DEV), off, wq.to(DEV), wsc.to(DEV),
                                      g.reshape(-1), y, ws)
    bits = moe.moe_check_status(ws)
    assert bits == 0, f"device status {bits:#x}"
    return bf16_np(y[:rows])


def _ref(which, offsets, aq, asc, wq, wsc, gs):
    g = gs.numpy() if which == "w13" else gs.numpy().reshape(-1)
    return o.grouped_gemm(aq.numpy(), asc.numpy(), offsets, wq.numpy(), wsc.numpy(),
                          fmt="nvfp4", w_global=g)


NV_SHAPES = [
    ("w13", 3, 512, 512, [5, 0, 11]),                 # small
    ("w2", 2, 512, 256, [1, 2]),
    ("w13", 4, 512, 1024, [16, 17, 33, 130]),         # small, medium, medium, large
    ("w2", 3, 256, 512, [300, 7, 128]),               # large (2 chunks), small, mid
    ("w13", 5, 512, 512, [0, 16, 64, 65, 129]),       # every boundary
    ("w13", 2, 512, 512, [224, 150]),                 # large
    # more small-group tiles than one wave of CTAs
    ("w13", 40, 1024, 768, [(i * 7) % 17 for i in range(40)]),
    ("w2", 24, 2048, 1536, [(i * 5) % 16 + 1 for i in range(24)]),
    # decode-like: long K, 1-7 rows per group
    ("w13", 6, 1024, 7168, [1, 2, 7, 1, 0, 3]),
    ("w13", 3, 512, 1024, [256, 100, 250]),           # mid chunks
    ("w13", 5, 512, 1024, [17, 32, 24, 33, 16]),      # medium tiles' lower range
    # small tiles whose last partial wave is split into K parts (on 152 SMs: 160 tiles ->
    # 8 tiles in 4 parts; 212 tiles -> 60 tiles in 2 parts; long K in 4 parts)
    ("w13", 20, 1024, 1024, [(i % 16) + 1 for i in range(20)]),
    ("w2", 53, 512, 3072, [(i * 3) % 16 + 1 for i in range(53)]),
    ("w13", 40, 512, 7168, [1 + i % 7 for i in range(40)]),
    ("w2", 2, 1536, 1536, [200, 129]),
    ("w13", 3, 512, 7168, [224, 0, 190]),             # large, long K
    ("w2", 2, 512, 3072, [240, 241]),                 # 240-row chunk, then 2 of 121
]


@pytest.mark.parametrize("which,G,N,K,sizes", NV_SHAPES)
def test_nvfp4_gemm_exact_integer(which, G, N, K, sizes):
    case = _nv_case(which, G, N, K, sizes, seed=G * N + K, integer=True)
    y = _run_nv(which, G, N, K, *case)
    ref = _ref(which, *case)
    bad = np.argwhere(y != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}: " \
                          f"got {y[tuple(bad[0])]} want {ref[tuple(bad[0])]}"


@pytest.mark.parametrize("which,G,N,K,sizes", NV_SHAPES)
def test_nvfp4_gemm_random(which, G, N, K, sizes):
    case = _nv_case(which, G, N, K, sizes, seed=G + N + K, integer=False)
    y = _run_nv(which, G, N, K, *case)
    assert_float_close(y, _ref(which, *case), f"{which} y")


def test_nvfp4_gemm_scale_addressing():
    """One non-unit E4M3 block scale at a time (a 16-element block in the first and in
    the second half of a 256-K stage, rows in both 32-row quarters of the converter
    warps), and distinct gate / up tensor scales: bit-exact on integer inputs."""
    which, G, N, K, sizes = "w13", 2, 512, 768, [3, 20]
    offsets, aq, asc, wq, wsc, gs = _nv_case(which, G, N, K, sizes, seed=11, integer=True)
    wsc = torch.full_like(wsc, 0x38)
    wsc[0, 3, 0] = 0x40
    wsc[0, 77, 9] = 0x44
    wsc[1, 300, 47] = 0x40
    wsc[1, 511, 24] = 0x44
    gs = torch.tensor([[1.0, 2.0], [0.5, 1.0]], dtype=torch.float32)
    y = _run_nv(which, G, N, K, offsets, aq, asc, wq, wsc, gs)
    ref = _ref(which, offsets, aq, asc, wq, wsc, gs)
    assert np.array_equal(y, ref)


def test_nvfp4_gemm_gathered_rows():
    """moe_grouped_gemm_w13_nvfp4 with perm_src: packed rows gathered from the tokens'
    FP8 rows (routed rows then shared rows)."""
    d = gi.Dims(T=40, H=512, I=256, E=6, k=3, has_shared=1)
    t = gi.custom_layer(d, seed=4)
    nv = gi.nvfp4_layer_weights(d, seed=4)
    idx, _ = o.route(t["logits"].numpy(), d.k)
    counts, offsets, perm_src, inv = o.permute(idx, d.E, d.has_shared)
    xq, xs = o.quant_act(bits_np(t["x"]))
    md = moe.dims(d.T, d.H, d.I, d.E, d.k, d.has_shared)
    y = torch.empty(d.Rs, 2 * d.I, dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(moe.gemm_workspace_size_nvfp4(md))
    moe.moe_grouped_gemm_w13_nvfp4(md, torch.from_numpy(xq).to(DEV), torch.from_numpy(xs).to(DEV),
                                   torch.from_numpy(perm_src).to(DEV),
                                   torch.from_numpy(offsets).to(DEV), nv["w13"].to(DEV),
                                   nv["w13_s"].to(DEV), nv["w13_gs"].to(DEV), y, ws)
    assert moe.moe_check_status(ws) == 0
    tok = o.packed_row_token(perm_src, d.T, d.k, d.has_shared)
    ref = o.grouped_gemm(xq[tok], xs[tok], offsets, nv["w13"].numpy(), nv["w13_s"].numpy(),
                         fmt="nvfp4", w_global=nv["w13_gs"].numpy())
    assert_float_close(bf16_np(y), ref, "y13 gathered")


def _forward_nv(d, t, nv):
    md = moe.dims(d.T, d.H, d.I, d.E, d.k, d.has_shared)
    dbg = moe.debug_buffers(md)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(moe.workspace_size_nvfp4(md))
    moe.moe_forward_nvfp4(md, t["x"].to(DEV), t["logits"].to(DEV), nv["w13"].to(DEV),
                          nv["w13_s"].to(DEV), nv["w13_gs"].to(DEV), nv["w2"].to(DEV),
                          nv["w2_s"].to(DEV), nv["w2_gs"].to(DEV), out, ws, debug=dbg)
    bits = moe.moe_check_status(ws)
    assert bits == 0, f"device status {bits:#x}"
    return out, {k: v.cpu() for k, v in dbg.items()}


@pytest.mark.parametrize("T,H,I,E,k,sh,kind", [
    (64, 512, 256, 8, 2, 0, "gate"),      # the tiny workload's shapes
    (37, 768, 512, 12, 4, 1, "normal"),   # ragged, shared expert
    (300, 256, 256, 5, 2, 1, "zipf"),     # groups past 128 rows: mid and large tiles
])
def test_forward_nvfp4_matches_oracle(T, H, I, E, k, sh, kind):
    d = gi.Dims(T=T, H=H, I=I, E=E, k=k, has_shared=sh)
    t = with_gate_logits(gi.custom_layer(d, seed=T, logits_kind=kind))
    nv = gi.nvfp4_layer_weights(d, seed=T)
    out, g = _forward_nv(d, t, nv)
    ref = o.moe_forward(bits_np(t["x"]), t["logits"].cpu().numpy(), d.k, nv["w13"].numpy(),
                        nv["w13_s"].numpy(), nv["w2"].numpy(), nv["w2_s"].numpy(), d.has_shared,
                        "nvfp4", nv["w13_gs"].numpy(), nv["w2_gs"].numpy())
    R = d.T * d.k
    for name in ("idx", "counts", "offsets", "xq", "xs"):
        assert np.array_equal(g[name].numpy(), ref[name]), name
    assert np.array_equal(g["perm_src"].numpy()[:R], ref["perm_src"])
    assert np.array_equal(g["inv"].numpy()[:R], ref["inv"])
    assert_float_close(bf16_np(g["y13"]), ref["y13"], "y13")
    assert_fp8_codes_close(g["hq"].numpy(), g["hs"].numpy(), ref["hq"], ref["hs"], "hq")
    assert_float_close(bf16_np(g["y2"]), ref["y2"], "y2")
    assert_float_close(bf16_np(out), ref["out"], "out")


def test_forward_nvfp4_decode_full_size_sampled():
    """The decode workload (T=7, H=7168, I=3072, 384 experts + shared) with NVFP4
    weights: integer stages in full, two whole tokens through the oracle."""
    d, t = gi.make_layer("decode", seed=0, device=DEV)
    del t["w13"], t["w13_s"], t["w2"], t["w2_s"]
    nv = gi.nvfp4_layer_weights(d, seed=0, device=DEV)
    out, g = _forward_nv(d, t, nv)
    lg = t["logits"].cpu().numpy()
    ridx, _ = o.route(lg, d.k)
    assert np.array_equal(g["idx"].numpy(), ridx)
    xq, xs = o.quant_act(bits_np(t["x"]))
    assert np.array_equal(g["xq"].numpy(), xq) and np.array_equal(g["xs"].numpy(), xs)
    toks = np.array([1, 5])
    experts = sorted(set(ridx[toks].ravel().tolist()) | {d.E})
    w = {n: np.zeros((d.G,) + tuple(nv[n].shape[1:]), np.uint8)
         for n in ("w13", "w13_s", "w2", "w2_s")}
    for e in experts:
        for n in w:
            w[n][e] = nv[n][e].cpu().numpy()
    ref = o.moe_forward_tokens(bits_np(t["x"]), lg, d.k, w["w13"], w["w13_s"], w["w2"],
                               w["w2_s"], d.has_shared, toks, "nvfp4",
                               nv["w13_gs"].cpu().numpy(), nv["w2_gs"].cpu().numpy())
    assert_float_close(bf16_np(out[torch.from_numpy(toks).to(DEV)]), ref["out"], "out")
    del t, nv
    torch.cuda.empty_cache()
