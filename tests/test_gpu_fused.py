"""GPU parity of the fusion and tile options through moe_forward_ex.

f2 (the weighted top-k combine + shared-expert add performed by the W2 GEMM's
epilogue; LMSYS-H20 §3.2) and f1 (SwiGLU + FP8 quantisation performed by the W13 GEMM's
epilogue on SM pairs; LMSYS-H20 §4.3) must reproduce the stand-alone path bit for bit
(the same fp32 arithmetic in the same order), across every GEMM tile variant, and match
the oracle.  The SM-pair tiles for groups above 64 rows must be bit-exact on
exact-integer inputs and within the float contract otherwise."""

import numpy as np
import pytest
import torch

import moe_expert_ffn_scan_gb300 as moe
from gen import inputs as gi
from oracle import moe_oracle as o
from tests._parity import assert_float_close, bf16_np, bits_np, with_gate_logits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(d, t, fuse_combine=False, fuse_swiglu=False, pair_tiles=False, more=False,
         large_chunk_rows=0):
    md = moe.dims(d.T, d.H, d.I, d.E, d.k, d.has_shared)
    out = torch.full((d.T, d.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(moe.workspace_size(md))
    dbg = {"y2": torch.empty(d.Rs, d.H, dtype=torch.bfloat16, device=DEV)}
    if more:
        dbg.update(hq=torch.empty(d.Rs, d.I, dtype=torch.uint8, device=DEV),
                   hs=torch.empty(d.Rs, d.I // 128, dtype=torch.uint8, device=DEV),
                   y13=torch.empty(d.Rs, 2 * d.I, dtype=torch.bfloat16, device=DEV))
    moe.moe_forward_ex(md, t["x"], t["logits"], t["w13"], t["w13_s"], t["w2"], t["w2_s"], out, ws,
                       fuse_combine=fuse_combine, fuse_swiglu=fuse_swiglu, pair_tiles=pair_tiles,
                       large_chunk_rows=large_chunk_rows, debug=dbg)
    bits = moe.moe_check_status(ws)
    assert bits == 0, f"device status {bits:#x}"
    return (out, dbg["y2"]) if not more else (out, dbg)


@pytest.mark.parametrize("T,H,I,E,k,sh,kind", [
    (64, 512, 256, 8, 2, 0, "gate"),      # the tiny workload: no shared expert
    (37, 768, 384, 12, 4, 1, "normal"),   # ragged, shared expert
    (7, 1024, 256, 64, 8, 1, "normal"),   # decode-like: 1-2 rows per group, small tiles
    (300, 256, 256, 5, 2, 1, "zipf"),     # groups past 128 rows: mid and large tiles
    (1000, 512, 256, 16, 6, 1, "zipf"),   # many tiles per token, every variant
    (96, 256, 256, 24, 12, 1, "normal"),  # top-k past 8: the gather's second row batch
    (40, 512, 256, 16, 16, 0, "normal"),  # top-16 of 16: every token in every group
])
def test_fused_combine_equals_standalone(T, H, I, E, k, sh, kind):
    d = gi.Dims(T=T, H=H, I=I, E=E, k=k, has_shared=sh)
    t = {n: (v.to(DEV) if v is not None else None)
         for n, v in with_gate_logits(gi.custom_layer(d, seed=T, logits_kind=kind)).items()}
    ref_out, ref_y2 = _run(d, t)
    out, y2 = _run(d, t, fuse_combine=True)
    assert torch.equal(y2, ref_y2)
    assert torch.equal(out, ref_out), int((out != ref_out).sum())
    # and the oracle's combine of the same y2 rows
    inv = o.permute(o.route(t["logits"].cpu().numpy(), k)[0], E, sh)[3]
    w = o.route(t["logits"].cpu().numpy(), k)[1]
    ref = o.combine(bf16_np(y2), inv, w, T, k, sh)
    assert_float_close(bf16_np(out), ref, "out")


def test_fused_combine_repeated_calls():
    """The arrival counters are reset by every forward: three calls in a row agree."""
    d = gi.Dims(T=200, H=512, I=256, E=10, k=4, has_shared=1)
    t = {n: (v.to(DEV) if v is not None else None)
         for n, v in gi.custom_layer(d, seed=5, logits_kind="zipf").items()}
    first, _ = _run(d, t, fuse_combine=True)
    for _ in range(2):
        again, _ = _run(d, t, fuse_combine=True)
        assert torch.equal(again, first)


@pytest.mark.parametrize("T,H,I,E,k,sh,kind", [
    (64, 512, 256, 8, 2, 0, "gate"),      # the tiny workload's shapes
    (37, 1024, 384, 12, 4, 1, "normal"),  # I/128 odd: the pair tiles cover 3 blocks
    (7, 1024, 256, 64, 8, 1, "normal"),   # decode-like: 1-2 rows per group
    (300, 512, 256, 5, 2, 1, "zipf"),     # groups past 128 rows: every plan list
    (900, 512, 512, 16, 6, 1, "zipf"),    # many tiles, chunks of up to 224 rows
])
def test_fused_swiglu_equals_standalone(T, H, I, E, k, sh, kind):
    d = gi.Dims(T=T, H=H, I=I, E=E, k=k, has_shared=sh)
    t = {n: (v.to(DEV) if v is not None else None)
         for n, v in with_gate_logits(gi.custom_layer(d, seed=T + 1, logits_kind=kind)).items()}
    ref_out, ref = _run(d, t, more=True)
    out, got = _run(d, t, fuse_swiglu=True, more=True)
    for n in ("hq", "hs"):
        bad = int((got[n] != ref[n]).sum())
        assert bad == 0, f"{n}: {bad} differing bytes"
    assert torch.equal(got["y2"], ref["y2"])
    assert torch.equal(out, ref_out)
    # and against the oracle's quantisation of the stand-alone path's y13
    rq, rs = o.swiglu_quant(bf16_np(ref["y13"]))
    assert np.array_equal(got["hs"].cpu().numpy(), rs) or \
        np.mean(got["hs"].cpu().numpy() != rs) < 1e-3


def test_pair_tiles_exact_integer_y13():
    """Groups above 64 rows on SM pairs: integer activations (x in {-8..8}, so every FP8
    code is exact) and integer MXFP4 weights with unit scales make every y13 an exact
    integer, equal to the oracle's."""
    d = gi.Dims(T=600, H=1024, I=256, E=6, k=2, has_shared=1)
    t = gi.custom_layer(d, seed=9, logits_kind="zipf")
    g = torch.Generator().manual_seed(9)
    t["x"] = torch.randint(-8, 9, (d.T, d.H), generator=g).to(torch.bfloat16)
    t["w13"] = gi.integer_fp4_bytes((d.G, 2 * d.I, d.H // 2), 9, "cpu", "w13")
    t["w13_s"] = torch.full((d.G, 2 * d.I, d.H // 32), 127, dtype=torch.uint8)
    td = {n: (v.to(DEV) if v is not None else None) for n, v in t.items()}
    _, got = _run(d, td, pair_tiles=True, more=True)
    ref = o.moe_forward(bits_np(t["x"]), t["logits"].numpy(), d.k, t["w13"].numpy(),
                        t["w13_s"].numpy(), t["w2"].numpy(), t["w2_s"].numpy(), d.has_shared)
    y13 = bf16_np(got["y13"])
    bad = np.argwhere(y13 != ref["y13"])
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("pair", [True, False])
def test_exact_integer_y13_at_chunk_boundaries(pair):
    """Groups of exactly 128, 129, 240, 256, 480 and 512 rows (one-hot logits, top-1):
    one mid chunk, one large chunk of 129 rows, two mid chunks of 120 / 128, three large
    chunks of 160 and of 171 rows -- on SM pairs and on one SM, y13 equal to the
    oracle's exact integers (integer activations, integer E2M1 codes, unit scales)."""
    sizes = [128, 129, 240, 256, 480, 512]
    E, T = len(sizes), sum(sizes)
    d = gi.Dims(T=T, H=1024, I=256, E=E, k=1, has_shared=0)
    t = gi.custom_layer(d, seed=21, logits_kind="normal")
    expert = np.repeat(np.arange(E), sizes)
    logits = torch.full((T, E), -8.0, dtype=torch.float32)
    logits[torch.arange(T), torch.from_numpy(expert)] = 8.0
    t["logits"] = logits
    g = torch.Generator().manual_seed(21)
    t["x"] = torch.randint(-8, 9, (d.T, d.H), generator=g).to(torch.bfloat16)
    t["w13"] = gi.integer_fp4_bytes((d.G, 2 * d.I, d.H // 2), 21, "cpu", "w13")
    t["w13_s"] = torch.full((d.G, 2 * d.I, d.H // 32), 127, dtype=torch.uint8)
    td = {n: (v.to(DEV) if v is not None else None) for n, v in t.items()}
    _, got = _run(d, td, pair_tiles=pair, more=True)
    ref = o.moe_forward(bits_np(t["x"]), t["logits"].numpy(), d.k, t["w13"].numpy(),
                        t["w13_s"].numpy(), t["w2"].numpy(), t["w2_s"].numpy(), d.has_shared)
    y13 = bf16_np(got["y13"])
    bad = np.argwhere(y13 != ref["y13"])
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("T,kind", [(300, "zipf"), (2000, "zipf")])
def test_pair_tiles_forward_matches_oracle(T, kind):
    d = gi.Dims(T=T, H=1024, I=512, E=8, k=4, has_shared=1)
    t = {n: (v.to(DEV) if v is not None else None)
         for n, v in gi.custom_layer(d, seed=T + 2, logits_kind=kind).items()}
    out, got = _run(d, t, pair_tiles=True, more=True)
    ref_out, ref = _run(d, t, more=True)
    assert_float_close(bf16_np(got["y13"]), bf16_np(ref["y13"]), "y13 (pair vs one SM)")
    assert_float_close(bf16_np(out), bf16_np(ref_out), "out (pair vs one SM)")


@pytest.mark.parametrize("pair", [False, True])
def test_chunk_rows_give_identical_outputs(pair):
    """The tile plan's chunk size (exact-shape tuning, LMSYS-H20 §3.3) changes only how
    groups above 64 rows are tiled (mid vs large tiles, chunk boundaries): every output
    element's K sum runs in the same order, so y13, hq/hs, y2 and out are equal bit for
    bit to the default plan's.  Zipf groups of up to ~1000 rows."""
    d = gi.Dims(T=2000, H=512, I=256, E=16, k=6, has_shared=1)
    t = {n: (v.to(DEV) if v is not None else None)
         for n, v in gi.custom_layer(d, seed=11, logits_kind="zipf").items()}
    ref_out, ref = _run(d, t, pair_tiles=pair, more=True)
    for c in (144, 160, 176, 208):
        out, got = _run(d, t, pair_tiles=pair, more=True, large_chunk_rows=c)
        for n in ("y13", "hq", "hs", "y2"):
            assert torch.equal(got[n], ref[n]), (c, n)
        assert torch.equal(out, ref_out), c


def test_chunk_rows_tuner_returns_a_candidate():
    d = gi.Dims(T=1024, H=512, I=256, E=8, k=4, has_shared=1)
    t = {n: (v.to(DEV) if v is not None else None)
         for n, v in gi.custom_layer(d, seed=12, logits_kind="zipf").items()}
    layer = moe.MoELayer(d.H, d.I, d.E, d.k, d.has_shared, t["w13"], t["w13_s"], t["w2"],
                         t["w2_s"])
    ref = layer.forward(t["x"], t["logits"]).clone()
    best, times = layer.tune_chunk_rows(t["x"], t["logits"], candidates=(224, 176, 144),
                                        steps=3, warmup=1)
    assert best in (224, 176, 144) and set(times) == {224, 176, 144}
    assert layer.large_chunk_rows == best
    assert torch.equal(layer.forward(t["x"], t["logits"]), ref)
    assert moe.moe_check_status(layer.workspace(d.T)) == 0


def test_options_are_validated():
    import ctypes
    d = moe.dims(7, 512, 256, 8, 2, 0)
    W = moe.moe_weights(0x10000, 0x10000, 0x10000, 0x10000)
    opt = moe.moe_options(2, 0, 0)
    P = ctypes.c_void_p
    assert moe.lib().moe_forward_ex(ctypes.byref(d), P(0x1000), P(0x1000), ctypes.byref(W),
                                    ctypes.byref(opt), P(0x1000), None, None, P(0x10000), 1 << 30,
                                    None) == 1
