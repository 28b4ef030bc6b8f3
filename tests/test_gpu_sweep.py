"""Grouped-GEMM sweep shapes at full size (W13: N=6144, K=7168; W2: N=7168, K=3072),
through the C interface, checked on sampled rows and output columns that the oracle
computes one by one from the same seeded inputs."""

import numpy as np
import pytest
import torch

import moe_expert_ffn_scan_gb300 as moe
from gen import inputs as gi
from oracle import moe_oracle as o
from tests._parity import assert_float_close, bf16_np, bits_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.mark.parametrize("which,M", [("w13", 1), ("w13", 7), ("w2", 16), ("w13", 32),
                                     ("w2", 32), ("w13", 64), ("w2", 512), ("w13", 4096),
                                     ("w2", 2048)])
def test_sweep_point_sampled(which, M):
    N, K = gi.SWEEP_SHAPES[which]
    G = min(gi.sweep_groups(M), 32)  # fewer groups than the bench sweep: same per-group work
    x, offsets, w, ws_ = gi.sweep_point(which, M, seed=M, device=DEV, G=G)
    rows = x.shape[0]
    q = torch.empty(rows, K, dtype=torch.uint8, device=DEV)
    qs = torch.empty(rows, K // 128, dtype=torch.uint8, device=DEV)
    moe.moe_quant_act(x, q, qs)
    y = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
    d = moe.dims(rows, K, N // 2, G, 1, 0) if which == "w13" else moe.dims(rows, N, K, G, 1, 0)
    wsp = moe.alloc_workspace(moe.gemm_workspace_size(d))
    if which == "w13":
        moe.moe_grouped_gemm_w13(d, q, qs, None, offsets, w, ws_, y, wsp)
    else:
        moe.moe_grouped_gemm_w2(d, q, qs, offsets, w, ws_, y, wsp)
    assert moe.moe_check_status(wsp) == 0
    rng = np.random.default_rng(M)
    r_s = np.unique(rng.choice(rows, size=min(rows, 24), replace=False))
    n_s = np.unique(rng.choice(N, size=96, replace=False))
    # the oracle quantises the same bf16 rows itself (bit-exact with the library's codes)
    aq, asc = o.quant_act(bits_np(x[torch.from_numpy(r_s).to(DEV)]))
    assert np.array_equal(aq, q[torch.from_numpy(r_s).to(DEV)].cpu().numpy())
    g_of_row = np.searchsorted(offsets.cpu().numpy(), r_s, side="right") - 1
    ref = np.empty((len(r_s), len(n_s)))
    for gi_ in np.unique(g_of_row):
        sel = np.where(g_of_row == gi_)[0]
        wg = w[int(gi_)][torch.from_numpy(n_s).to(DEV)].cpu().numpy()[None]
        wsg = ws_[int(gi_)][torch.from_numpy(n_s).to(DEV)].cpu().numpy()[None]
        off = np.array([0, len(sel)], np.int32)
        ref[sel] = o.grouped_gemm(aq[sel], asc[sel], off, wg, wsg)
    got = bf16_np(y[torch.from_numpy(r_s).to(DEV)][:, torch.from_numpy(n_s).to(DEV)])
    assert_float_close(got, ref, f"{which} M={M}")
