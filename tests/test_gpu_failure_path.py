"""The device failure path, exercised without a GPU fault: a wait that nothing will
ever complete must give up after the library's bound (2 s of the GPU's global timer),
report STATUS_WAIT_TIMEOUT through the workspace status word, and leave the context
usable for the next layer."""

import pytest
import torch

import moe_expert_ffn_scan_gb300 as moe
from gen import inputs as gi
from tests._parity import with_gate_logits

pytestmark = pytest.mark.gpu

STATUS_WAIT_TIMEOUT = 1 << 0


def test_bounded_wait_times_out_and_context_survives():
    ws = moe.alloc_workspace(256)
    moe.moe_selftest_wait_timeout(ws)
    bits = moe.moe_check_status(ws)  # synchronises
    assert bits == STATUS_WAIT_TIMEOUT, f"status {bits:#x}"
    # the context still runs a layer, and the layer's own status word is clean
    d, t = gi.make_layer("tiny", device="cuda")
    with_gate_logits(t)
    layer = moe.MoELayer(d.H, d.I, d.E, d.k, d.has_shared, t["w13"], t["w13_s"], t["w2"],
                         t["w2_s"])
    out = layer.forward(t["x"], t["logits"])
    torch.cuda.synchronize()
    assert moe.moe_check_status(layer.workspace(d.T)) == 0
    assert torch.isfinite(out.float()).all()
