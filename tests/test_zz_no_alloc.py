"""moe_route_static: routing for callers that cannot allocate device memory.

Some callers may not call cudaMalloc at all -- a host framework whose memory pool
owns every device byte, or a latency-critical loop that cannot pay for cudaMalloc /
cudaFree and the device synchronisation they can cause.  moe_route_static gives
them the routing + permutation call with its scratch in a fixed array inside the
library.  This test calls it through the C interface twice in a row (the array
keeps the previous call's contents) and checks every output against moe_route,
which uses a caller workspace.  Kept in a file of its own, collected last."""

import ctypes

import numpy as np
import pytest
import torch

import moe_expert_ffn_scan_gb300 as moe
from gen import inputs as gi

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _outputs(d):
    T, E, k, sh = d.T, d.E, d.k, d.has_shared
    return dict(idx=torch.empty(T, k, dtype=torch.int32, device=DEV),
                w=torch.empty(T, k, dtype=torch.float32, device=DEV),
                counts=torch.empty(E, dtype=torch.int32, device=DEV),
                offsets=torch.empty(E + sh + 1, dtype=torch.int32, device=DEV),
                perm_src=torch.full((T * k,), -7, dtype=torch.int32, device=DEV),
                inv=torch.full((T * k,), -7, dtype=torch.int32, device=DEV))


def _route_static(d, logits):
    L = moe.lib()
    fn = L.moe_route_static
    P = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(moe.moe_dims)] + [P] * 8
    fn.restype = ctypes.c_int
    o = _outputs(d)
    rc = fn(ctypes.byref(d), P(logits.data_ptr()), *[P(o[n].data_ptr()) for n in
            ("idx", "w", "counts", "offsets", "perm_src", "inv")],
            P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, f"moe_route_static returned {rc}"
    return o


def _route_ws(d, logits):
    o = _outputs(d)
    ws = moe.alloc_workspace(moe.route_workspace_size(d))
    moe.moe_route(d, logits, o["idx"], o["w"], o["counts"], o["offsets"], o["perm_src"],
                  o["inv"], ws)
    assert moe.moe_check_status(ws) == 0
    return o


def _static_status():
    fn = moe.lib().moe_route_static_status
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    fn.restype = ctypes.c_int
    bits = ctypes.c_uint32(0xFFFFFFFF)
    rc = fn(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(bits))
    assert rc in (0, 5), rc
    return bits.value


def test_route_static_matches_route_two_calls_in_a_row():
    cases = [(moe.dims(4096, 128, 128, 384, 8, 1), "zipf", 1),
             (moe.dims(7, 128, 128, 384, 8, 1), "normal", 2)]
    for d, kind, seed in cases:
        lg = (gi.zipf_logits(d.T, d.E, seed, "cpu") if kind == "zipf" else
              torch.randn(d.T, d.E, generator=torch.Generator().manual_seed(seed))).to(DEV)
        got = _route_static(d, lg)
        ref = _route_ws(d, lg)
        torch.cuda.synchronize()
        for n in ("idx", "counts", "offsets", "perm_src", "inv"):
            assert torch.equal(got[n], ref[n]), n
        # same kernels on the same inputs: the weights agree bit for bit too, well
        # inside the float tolerance the other tests use (rtol 2e-6)
        np.testing.assert_allclose(got["w"].cpu().numpy(), ref["w"].cpu().numpy(), rtol=2e-6)
        # the device-side index checks of the call found nothing
        assert _static_status() == 0


def test_route_static_rejects_sizes_beyond_its_scratch():
    fn = moe.lib().moe_route_static
    P = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(moe.moe_dims)] + [P] * 8
    fn.restype = ctypes.c_int
    d = moe.dims(8193, 128, 128, 1024, 8, 0)   # ceil(8193/256) * 1024 > 32768
    assert fn(ctypes.byref(d), *[P(0x1000)] * 7, None) == 2
    # a misaligned pointer is rejected on the host, before any launch
    d = moe.dims(64, 128, 128, 8, 2, 0)
    assert fn(ctypes.byref(d), P(0x1002), *[P(0x1000)] * 6, None) == 1
    assert fn(ctypes.byref(d), P(0x1000), P(0x1000), P(0x1001), *[P(0x1000)] * 4, None) == 1


def test_route_static_survives_device_reset():
    """After cudaDeviceReset the library's module, and the fixed array with it, is
    loaded again, possibly elsewhere: the array's address is looked up again in the new
    context.  Run in a child process, whose context the reset may end."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, os.path.join(here, "_route_static_reset_child.py")],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
