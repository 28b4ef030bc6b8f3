"""GPU parity of the fusion options (f2: the weighted top-k combine + shared-expert add
performed by the W2 GEMM's epilogue; LMSYS-H20 §3.2) through moe_forward_ex: the
fused layer's output must equal the stand-alone path's bit for bit (same fp32 sums in
the same order), across every GEMM tile variant, and match the oracle."""

import numpy as np
import pytest
import torch

import moe_expert_ffn_scan_gb300 as moe
from gen import inputs as gi
from oracle import moe_oracle as o
from tests._parity import assert_float_close, bf16_np, bits_np, with_gate_logits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(d, t, fuse_combine):
    md = moe.dims(d.T, d.H, d.I, d.E, d.k, d.has_shared)
    out = torch.full((d.T, d.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(moe.workspace_size(md))
    dbg = {"y2": torch.empty(d.Rs, d.H, dtype=torch.bfloat16, device=DEV)}
    moe.moe_forward_ex(md, t["x"], t["logits"], t["w13"], t["w13_s"], t["w2"], t["w2_s"], out, ws,
                       fuse_combine=fuse_combine, debug=dbg)
    bits = moe.moe_check_status(ws)
    assert bits == 0, f"device status {bits:#x}"
    return out, dbg["y2"]


@pytest.mark.parametrize("T,H,I,E,k,sh,kind", [
    (64, 512, 256, 8, 2, 0, "gate"),      # the tiny workload: no shared expert
    (37, 768, 384, 12, 4, 1, "normal"),   # ragged, shared expert
    (7, 1024, 256, 64, 8, 1, "normal"),   # decode-like: 1-2 rows per group, small tiles
    (300, 256, 256, 5, 2, 1, "zipf"),     # groups past 128 rows: mid and large tiles
    (1000, 512, 256, 16, 6, 1, "zipf"),   # many tiles per token, every variant
])
def test_fused_combine_equals_standalone(T, H, I, E, k, sh, kind):
    d = gi.Dims(T=T, H=H, I=I, E=E, k=k, has_shared=sh)
    t = {n: (v.to(DEV) if v is not None else None)
         for n, v in with_gate_logits(gi.custom_layer(d, seed=T, logits_kind=kind)).items()}
    ref_out, ref_y2 = _run(d, t, False)
    out, y2 = _run(d, t, True)
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
    first, _ = _run(d, t, True)
    for _ in range(2):
        again, _ = _run(d, t, True)
        assert torch.equal(again, first)


def test_options_are_validated():
    import ctypes
    d = moe.dims(7, 512, 256, 8, 2, 0)
    W = moe.moe_weights(0x10000, 0x10000, 0x10000, 0x10000)
    opt = moe.moe_options(2)
    P = ctypes.c_void_p
    assert moe.lib().moe_forward_ex(ctypes.byref(d), P(0x1000), P(0x1000), ctypes.byref(W),
                                    ctypes.byref(opt), P(0x1000), None, None, P(0x10000), 1 << 30,
                                    None) == 1
