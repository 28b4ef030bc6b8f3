"""GPU parity of the whole layer (moe_forward) against the oracle.

Small shapes are checked in full, stage by stage, on identical seeded inputs.  The
full-size decode and prefill workloads are checked on every integer output in full
and on sampled floating-point outputs that the oracle computes one by one."""

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


def _forward(d, t):
    dbg = moe.debug_buffers(d)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(moe.workspace_size(d))
    moe.moe_forward(d, t["x"], t["logits"], t["w13"], t["w13_s"], t["w2"], t["w2_s"], out, ws,
                    debug=dbg)
    bits = moe.moe_check_status(ws)
    assert bits == 0, f"device status {bits:#x}"
    return out, dbg


def _np(t):
    return {k: (v.cpu().numpy() if v.dtype != torch.bfloat16 else bits_np(v))
            for k, v in t.items() if v is not None}


def _check_full(d, t):
    out, dbg = _forward(d, {k: v.to(DEV) for k, v in t.items() if v is not None})
    n = _np(t)
    ref = o.moe_forward(n["x"], n["logits"], d.k, n["w13"], n["w13_s"], n["w2"], n["w2_s"],
                        d.has_shared)
    g = {k: v.cpu() for k, v in dbg.items()}
    R = d.T * d.k
    for name in ("idx", "counts", "offsets", "xq", "xs"):
        assert np.array_equal(g[name].numpy(), ref[name]), name
    assert np.array_equal(g["perm_src"].numpy()[:R], ref["perm_src"])
    assert np.array_equal(g["inv"].numpy()[:R], ref["inv"])
    np.testing.assert_allclose(g["w"].numpy(), ref["w"], rtol=2e-6, atol=1e-7)
    stats = {}
    stats["y13"] = assert_float_close(bf16_np(g["y13"]), ref["y13"], "y13")
    stats["hq_agree"] = assert_fp8_codes_close(g["hq"].numpy(), g["hs"].numpy(), ref["hq"],
                                               ref["hs"], "hq")
    stats["y2"] = assert_float_close(bf16_np(g["y2"]), ref["y2"], "y2")
    stats["out"] = assert_float_close(bf16_np(out), ref["out"], "out")
    return stats


def test_forward_tiny_workload():
    d, t = gi.make_layer("tiny")
    with_gate_logits(t)
    _check_full(moe.dims(d.T, d.H, d.I, d.E, d.k, d.has_shared), t)


@pytest.mark.parametrize("T,H,I,E,k,sh,kind", [
    (13, 256, 128, 5, 3, 1, "normal"),      # ragged, shared expert
    (1, 512, 256, 8, 2, 1, "normal"),       # a single token
    (200, 384, 256, 16, 4, 1, "zipf"),      # skewed: large and empty groups
    (40, 1024, 512, 64, 8, 0, "zipf"),
    (90, 256, 256, 3, 3, 0, "normal"),      # k == E: every token to every expert
    (128, 256, 128, 16, 4, 1, "zipf"),      # largest T of the one-CTA decode prep
    (129, 256, 128, 16, 4, 1, "zipf"),      # smallest T of the multi-kernel route path
    (5, 128, 128, 1, 1, 0, "normal"),       # one expert, k = 1, minimal H and I
    (3, 256, 128, 1024, 16, 1, "normal"),   # largest E and k the interface accepts
    (300, 640, 384, 12, 2, 1, "zipf"),      # H/128 and I/128 odd: one-sub-tile stages
])
def test_forward_ragged_shapes(T, H, I, E, k, sh, kind):
    d = gi.Dims(T=T, H=H, I=I, E=E, k=k, has_shared=sh)
    t = gi.custom_layer(d, seed=T + E, logits_kind=kind)
    _check_full(moe.dims(T, H, I, E, k, sh), t)


@pytest.mark.parametrize("workload", ["tiny", "decode"])
def test_forward_host_equals_device_forward(workload):
    """moe_forward_host (pinned host buffers in and out) gives the device forward's
    output bit for bit."""
    d, t = gi.make_layer(workload, seed=4, device=DEV)
    with_gate_logits(t)
    layer = moe.MoELayer(d.H, d.I, d.E, d.k, d.has_shared, t["w13"], t["w13_s"], t["w2"],
                         t["w2_s"])
    ref = layer.forward(t["x"], t["logits"])
    xh = t["x"].cpu().pin_memory()
    lgh = t["logits"].cpu().pin_memory()
    oh = torch.full((d.T, d.H), float("nan"), dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xh, lgh, oh)
    torch.cuda.synchronize()
    assert torch.equal(oh, ref.cpu())
    assert moe.moe_check_status(layer.host_workspace(d.T)) == 0
    hg = layer.host_graph(d.T)
    hg.x_host.copy_(xh)
    hg.logits_host.copy_(lgh)
    for _ in range(2):
        hg.out_host.fill_(float("nan"))
        hg.replay()
        torch.cuda.synchronize()
        assert torch.equal(hg.out_host, ref.cpu())


@pytest.mark.parametrize("workload,depth", [("tiny", 2), ("decode", 2), ("tiny", 1),
                                            ("tiny", 3)])
def test_host_pipeline_equals_device_forward(workload, depth):
    """Five steps with distinct inputs through the host-buffer pipeline (slots reused
    once depth steps are in flight): each output bit-identical to moe_forward on the
    same inputs."""
    d, t = gi.make_layer(workload, device=DEV)
    layer = moe.MoELayer(d.H, d.I, d.E, d.k, d.has_shared, t["w13"], t["w13_s"], t["w2"],
                         t["w2_s"])
    steps = 5
    xs = [gi.activations(d.T, d.H, 100 + i, DEV) for i in range(steps)]
    lgs = [gi.router_logits("normal", xs[i], d.E, 100 + i, DEV) for i in range(steps)]
    xh = [x.cpu().pin_memory() for x in xs]
    lh = [lg.cpu().pin_memory() for lg in lgs]
    oh = [torch.empty(d.T, d.H, dtype=torch.bfloat16).pin_memory() for _ in range(steps)]
    pipe = layer.host_pipeline(d.T, depth)
    for i in range(steps):
        pipe.submit(xh[i], lh[i], oh[i])
    pipe.sync()
    assert moe.moe_check_status(pipe.ws) == 0
    for i in range(steps):
        ref = layer.forward(xs[i], lgs[i])
        torch.cuda.synchronize()
        assert torch.equal(oh[i], ref.cpu()), f"step {i}"
    pipe.close()


def test_forward_zero_input():
    d, t = gi.make_layer("tiny")
    with_gate_logits(t)
    t["x"] = torch.zeros_like(t["x"])
    out, dbg = _forward(moe.dims(d.T, d.H, d.I, d.E, d.k, d.has_shared),
                        {k: v.to(DEV) for k, v in t.items() if v is not None})
    assert torch.all(out.float() == 0)


# ---------------------------------------------------------------- full size ---------

def _group_rows_at_tile_positions(offsets, G, rng, n_large=6, edge=720):
    """Packed rows to check: in every group its first and last row and two random ones;
    in the n_large largest groups also the rows on both sides of every 16-row boundary
    within `edge` rows of either end.  Groups above 240 rows are cut by the tile plan
    into near-equal chunks of multiples of 16 rows (mid variant up to 128, large up to
    240), so these rows land on every token-tile position of the first and last chunks,
    the ragged final chunk included."""
    sizes = np.diff(offsets[:G + 1])
    large = set(np.argsort(-sizes, kind="stable")[:n_large].tolist())
    rows = []
    for g in range(G):
        r0, m = int(offsets[g]), int(sizes[g])
        if m == 0:
            continue
        pos = {0, m - 1}
        pos.update(rng.integers(0, m, size=min(2, m)).tolist())
        if g in large:
            for b in range(16, m, 16):
                if b <= edge or b >= m - edge:
                    pos.update((b - 1, b))
        rows += [r0 + p for p in sorted(pos)]
    return np.array(sorted(set(rows)), dtype=np.int64)


def _packed_rows_check(d, t, dbg, offsets, perm_src, rows, n_cols, seed):
    """Stage-isolated checks of W13, SwiGLU + quant and W2 on the given packed rows:
    y13 against the oracle GEMM of the token's FP8 row with the group's weights, hq/hs
    against the oracle's quantisation of the GPU's own y13 row, and y2 against the
    oracle GEMM of the GPU's own hq/hs row; sampled output columns."""
    R = d.T * d.k
    rng = np.random.default_rng(seed)
    G = len(offsets) - 1
    grp = np.searchsorted(offsets, rows, side="right") - 1
    tok = np.where(rows < R, perm_src[np.minimum(rows, R - 1)] // d.k, rows - R)
    xq, xs = o.quant_act(bits_np(t["x"][torch.from_numpy(tok).to(DEV)]))
    sel = torch.from_numpy(rows).to(DEV)
    y13_rows = bf16_np(dbg["y13"][sel])
    hq_rows = dbg["hq"][sel].cpu().numpy()
    hs_rows = dbg["hs"][sel].cpu().numpy()
    y2_rows = bf16_np(dbg["y2"][sel])
    c13 = np.sort(rng.choice(2 * d.I, size=n_cols, replace=False))
    c2 = np.sort(rng.choice(d.H, size=n_cols, replace=False))
    ref13 = np.empty((len(rows), n_cols))
    ref2 = np.empty((len(rows), n_cols))
    for g in np.unique(grp):
        i = np.where(grp == g)[0]
        off = np.array([0, len(i)], np.int32)
        cc = torch.from_numpy(c13).to(DEV)
        ref13[i] = o.grouped_gemm(xq[i], xs[i], off, t["w13"][int(g)][cc].cpu().numpy()[None],
                                  t["w13_s"][int(g)][cc].cpu().numpy()[None])
        cc = torch.from_numpy(c2).to(DEV)
        ref2[i] = o.grouped_gemm(hq_rows[i], hs_rows[i], off,
                                 t["w2"][int(g)][cc].cpu().numpy()[None],
                                 t["w2_s"][int(g)][cc].cpu().numpy()[None])
    assert_float_close(y13_rows[:, c13], ref13, "y13 packed rows")
    rq, rs = o.swiglu_quant(y13_rows)
    assert_fp8_codes_close(hq_rows, hs_rows, rq, rs, "hq packed rows", max_mismatch=1e-3)
    assert_float_close(y2_rows[:, c2], ref2, "y2 packed rows")


def _sampled_check(workload, n_tokens, n_cols, seed=0):
    d, t = gi.make_layer(workload, seed=seed, device=DEV)
    md = moe.dims(d.T, d.H, d.I, d.E, d.k, d.has_shared)
    out, dbg = _forward(md, t)
    # integer stages in full
    lg = t["logits"].cpu().numpy()
    ridx, rw = o.route(lg, d.k)
    rc, roff, rperm, rinv = o.permute(ridx, d.E, d.has_shared)
    g = {k: v.cpu().numpy() for k, v in dbg.items() if v.dtype != torch.bfloat16}
    R = d.T * d.k
    assert np.array_equal(g["idx"], ridx)
    assert np.array_equal(g["counts"], rc)
    assert np.array_equal(g["offsets"], roff)
    assert np.array_equal(g["perm_src"][:R], rperm)
    assert np.array_equal(g["inv"][:R], rinv)
    np.testing.assert_allclose(g["w"], rw, rtol=2e-6, atol=1e-7)
    xbits = bits_np(t["x"])
    qrows = np.arange(d.T) if d.T <= 4096 else np.sort(
        np.random.default_rng(seed + 1).choice(d.T, 512, replace=False))
    xq, xs = o.quant_act(xbits[qrows])
    assert np.array_equal(g["xq"][qrows], xq) and np.array_equal(g["xs"][qrows], xs)
    # sampled floating-point outputs: whole tokens through the oracle
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(d.T, size=min(n_tokens, d.T), replace=False))
    experts = sorted(set(ridx[toks].ravel().tolist()) | ({d.E} if d.has_shared else set()))
    # the oracle sees the sampled tokens' rows and only the experts they use
    w13 = np.zeros((d.G,) + tuple(t["w13"].shape[1:]), np.uint8)
    w13s = np.zeros((d.G,) + tuple(t["w13_s"].shape[1:]), np.uint8)
    w2 = np.zeros((d.G,) + tuple(t["w2"].shape[1:]), np.uint8)
    w2s = np.zeros((d.G,) + tuple(t["w2_s"].shape[1:]), np.uint8)
    for e in experts:
        w13[e] = t["w13"][e].cpu().numpy()
        w13s[e] = t["w13_s"][e].cpu().numpy()
        w2[e] = t["w2"][e].cpu().numpy()
        w2s[e] = t["w2_s"][e].cpu().numpy()
    ref = o.moe_forward_tokens(xbits, lg, d.k, w13, w13s, w2, w2s, d.has_shared, toks)
    assert_float_close(bf16_np(out[torch.from_numpy(toks).to(DEV)]), ref["out"], "out")
    # y13 / y2 rows of the sampled tokens, sampled columns
    inv = g["inv"][:R].reshape(d.T, d.k)
    rows = np.concatenate([inv[toks].ravel()] + ([R + toks] if d.has_shared else []))
    ref_rows = np.concatenate([ref["inv"].reshape(len(toks), d.k).ravel()] +
                              ([len(toks) * d.k + np.arange(len(toks))] if d.has_shared else []))
    y13 = bf16_np(dbg["y13"][torch.from_numpy(rows).to(DEV)])
    assert_float_close(y13, ref["y13"][ref_rows], "y13 rows")
    y2 = bf16_np(dbg["y2"][torch.from_numpy(rows).to(DEV)])
    assert_float_close(y2, ref["y2"][ref_rows], "y2 rows")
    if n_cols:
        # packed rows at every tile position of every group (the largest groups reach
        # the mid and large GEMM variants), checked stage by stage on sampled columns
        prow = _group_rows_at_tile_positions(roff, d.G, np.random.default_rng(seed + 2))
        _packed_rows_check(d, t, dbg, roff, g["perm_src"], prow, n_cols, seed + 3)
    del t, dbg
    torch.cuda.empty_cache()


def test_forward_decode_full_size_sampled():
    _sampled_check("decode", n_tokens=2, n_cols=0)


def test_forward_decode256_full_size_sampled():
    _sampled_check("decode256", n_tokens=16, n_cols=64)


def test_forward_prefill_full_size_sampled():
    _sampled_check("prefill", n_tokens=1, n_cols=96)
