"""GPU parity of the router gate projection (moe_router_logits) against the oracle.

Bound: each logit is a sum of H products computed with fused multiply-adds in fp32
(the products are exact inside the FMA), so |got - exact| <= gamma_H * sum|x_h w_h|
with gamma_H = H u / (1 - H u), u = 2**-24, for any summation order; the oracle's
value is the exact sum rounded once to fp32 (another u * |sum|).  The test bound is
that sum of the two, element by element."""

import numpy as np
import pytest
import torch

import moe_expert_ffn_scan_gb300 as moe
from gen import inputs as gi
from oracle import moe_oracle as o
from tests._parity import bits_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
U = 2.0 ** -24


def _inputs(T, H, E, seed):
    x = gi.activations(T, H, seed, DEV)
    wg = gi.gate_weight(E, H, seed, DEV)
    return x, wg


def _bound(xb, wg):
    H = xb.shape[1]
    gamma = H * U / (1 - H * U)
    mag = np.abs(o.bf16_bits_to_f64(xb)) @ np.abs(wg.astype(np.float64)).T
    return (gamma + U) * mag


def _run(x, wg):
    lg = torch.full((x.shape[0], wg.shape[0]), float("nan"), dtype=torch.float32, device=DEV)
    moe.moe_router_logits(x, wg, lg)
    torch.cuda.synchronize()
    return lg


@pytest.mark.parametrize("T,H,E", [
    (7, 7168, 384),    # decode: the W_g-streaming kernel
    (1, 128, 8),
    (64, 512, 8),      # the tiny layer's dims
    (1024, 256, 24),   # largest T of the streaming kernel
    (1025, 512, 8),    # smallest T of the tiled kernel
    (130, 1024, 40),   # ragged token groups
    (1300, 256, 1000), # tiled: ragged token and expert tiles
    (16, 4096, 3),     # fewer experts than one CTA's share
    (17, 16, 7),       # H = one K stage
])
def test_router_logits_matches_oracle(T, H, E):
    x, wg = _inputs(T, H, E, seed=T + E)
    lg = _run(x, wg).cpu().numpy().astype(np.float64)
    xb = bits_np(x)
    wn = wg.cpu().numpy()
    ref = o.router_logits(xb, wn)
    err = np.abs(lg - ref)
    bound = _bound(xb, wn)
    assert np.all(np.isfinite(lg)), "unwritten or non-finite logits"
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{len(bad)} logits out of bound, first {bad[:3].tolist()}"
    # and typically far inside it (random-walk accumulation error)
    assert float(np.median(err / np.maximum(bound, 1e-300))) < 0.05


def test_router_logits_deterministic():
    x, wg = _inputs(300, 1024, 64, seed=5)
    a = _run(x, wg)
    b = _run(x, wg)
    assert torch.equal(a, b)
    x, wg = _inputs(7, 7168, 384, seed=5)
    assert torch.equal(_run(x, wg), _run(x, wg))
    x, wg = _inputs(2000, 512, 64, seed=5)  # the tiled kernel
    assert torch.equal(_run(x, wg), _run(x, wg))


def test_routing_of_projected_logits_matches_oracle():
    """Decode-sized gate: top-8 routing of the GPU logits equals the oracle routing of
    the oracle logits for every token whose top-9 oracle logits are separated by more
    than twice that token's largest GPU error (then GPU logit order = oracle order for
    them); tokens with closer logits are counted, not gated."""
    T, H, E, k = 64, 7168, 384, 8
    x, wg = _inputs(T, H, E, seed=11)
    lg = _run(x, wg)
    d = moe.dims(T, H, 3072, E, k, 0)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty(T * k, dtype=torch.int32, device=DEV)
    ws = moe.alloc_workspace(moe.route_workspace_size(d))
    moe.moe_route(d, lg, idx, w, counts, offsets, perm, inv, ws)
    xb, wn = bits_np(x), wg.cpu().numpy()
    ref = o.router_logits(xb, wn)
    ridx, _ = o.route(ref, k)
    err = np.abs(lg.cpu().numpy().astype(np.float64) - ref).max(axis=1)
    assert np.all(err <= _bound(xb, wn).max(axis=1))
    srt = np.sort(ref, axis=1)[:, ::-1]
    decidable = 0
    for t in range(T):
        if np.all(-np.diff(srt[t, :k + 1]) > 2 * err[t]):
            decidable += 1
            assert np.array_equal(idx[t].cpu().numpy(), ridx[t]), t
    assert decidable >= T // 2


def test_router_logits_prefill_size_sampled():
    """32K tokens x 7168 x 384 through the tiled kernel; 64 sampled tokens checked."""
    T, H, E = 32768, 7168, 384
    x, wg = _inputs(T, H, E, seed=0)
    lg = _run(x, wg)
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(T, size=64, replace=False))
    xb = bits_np(x[torch.from_numpy(toks).to(DEV)])
    wn = wg.cpu().numpy()
    ref = o.router_logits(xb, wn)
    got = lg[torch.from_numpy(toks).to(DEV)].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= _bound(xb, wn))
    assert torch.isfinite(lg).all()


# ---------------------------------------------------------------- tensor cores ------

def _run_split(x, wg):
    wg3 = moe.moe_router_split(wg)
    lg = torch.full((x.shape[0], wg.shape[0]), float("nan"), dtype=torch.float32, device=DEV)
    moe.moe_router_logits_split(x, wg3, lg)
    torch.cuda.synchronize()
    return lg, wg3


def test_router_split_is_exact():
    """hi + mid + lo reproduces every fp32 gate weight exactly (checked in float64)."""
    for E, H, seed in ((384, 7168, 1), (8, 512, 2)):
        wg = gi.gate_weight(E, H, seed, DEV)
        wg3 = moe.moe_router_split(wg)
        torch.cuda.synchronize()
        pieces = wg3.float().cpu().numpy().astype(np.float64)
        assert np.array_equal(pieces.sum(axis=0), wg.cpu().numpy().astype(np.float64))
    # and on values that need all three pieces: 24 significant bits
    w = torch.tensor([[1.0 + 2.0 ** -23, -3.0 - 2.0 ** -20, 0.02 + 2.0 ** -30, 1e-20] * 4],
                     dtype=torch.float32, device=DEV)
    p = moe.moe_router_split(w).float().cpu().numpy().astype(np.float64)
    assert np.array_equal(p.sum(axis=0), w.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("T,H,E", [
    (64, 512, 8),       # the tiny layer's dims: one tile, 8 of 128 expert columns
    (130, 1024, 40),    # ragged token tile
    (1300, 256, 1000),  # ragged token and expert tiles, many tiles per CTA
    (300, 7168, 384),   # the model's H and E
    (17, 16, 7),        # H below one 64-column stage
    (200, 80, 130),     # H not a multiple of 64: a zero-filled stage tail
])
def test_router_logits_split_matches_oracle(T, H, E):
    x, wg = _inputs(T, H, E, seed=T + E + 1)
    lg, _ = _run_split(x, wg)
    lg = lg.cpu().numpy().astype(np.float64)
    xb = bits_np(x)
    wn = wg.cpu().numpy()
    ref = o.router_logits(xb, wn)
    err = np.abs(lg - ref)
    bound = _bound(xb, wn)
    assert np.all(np.isfinite(lg)), "unwritten or non-finite logits"
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{len(bad)} logits out of bound, first {bad[:3].tolist()}"
    assert float(np.median(err / np.maximum(bound, 1e-300))) < 0.05


def test_router_logits_split_deterministic_and_prefill_sampled():
    T, H, E = 32768, 7168, 384
    x, wg = _inputs(T, H, E, seed=3)
    a, wg3 = _run_split(x, wg)
    b = torch.empty_like(a)
    moe.moe_router_logits_split(x, wg3, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(T, size=64, replace=False))
    xb = bits_np(x[torch.from_numpy(toks).to(DEV)])
    wn = wg.cpu().numpy()
    ref = o.router_logits(xb, wn)
    got = a[torch.from_numpy(toks).to(DEV)].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= _bound(xb, wn))
    assert torch.isfinite(a).all()
