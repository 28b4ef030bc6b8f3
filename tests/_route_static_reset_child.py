"""Child process of tests/test_zz_no_alloc.py::test_route_static_survives_device_reset.

Runs without torch's CUDA state (the device reset below would invalidate it): device
buffers come from the CUDA runtime through ctypes.  Calls moe_route_static, resets the
device (which ends this process's context and unloads the library's module), calls it
again, and checks both calls against moe_route with a caller workspace.  Prints "ok"."""

import ctypes
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import moe_expert_ffn_scan_gb300 as moe  # noqa: E402

P = ctypes.c_void_p
L = moe.lib()
rt = ctypes.CDLL("libcudart.so.13")
rt.cudaMalloc.argtypes = [ctypes.POINTER(P), ctypes.c_size_t]
rt.cudaMemcpy.argtypes = [P, P, ctypes.c_size_t, ctypes.c_int]
rt.cudaFree.argtypes = [P]
L.moe_route_static.argtypes = [ctypes.POINTER(moe.moe_dims)] + [P] * 8
L.moe_route_static.restype = ctypes.c_int
L.moe_route_static_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
L.moe_route_static_status.restype = ctypes.c_int


def check(rc, what):
    if rc != 0:
        raise SystemExit(f"{what} returned {rc}")


def dev_alloc(nbytes):
    p = P()
    check(rt.cudaMalloc(ctypes.byref(p), max(nbytes, 256)), "cudaMalloc")
    return p


def to_dev(a):
    p = dev_alloc(a.nbytes)
    check(rt.cudaMemcpy(p, a.ctypes.data_as(P), a.nbytes, 1), "cudaMemcpy h2d")
    return p


def to_host(p, shape, dtype):
    a = np.empty(shape, dtype)
    check(rt.cudaMemcpy(a.ctypes.data_as(P), p, a.nbytes, 2), "cudaMemcpy d2h")
    return a


def route(d, logits, static):
    T, E, k, sh = d.T, d.E, d.k, d.has_shared
    shapes = dict(idx=((T, k), np.int32), w=((T, k), np.float32), counts=((E,), np.int32),
                  offsets=((E + sh + 1,), np.int32), perm_src=((T * k,), np.int32),
                  inv=((T * k,), np.int32))
    lg = to_dev(logits)
    bufs = {n: dev_alloc(int(np.prod(s)) * np.dtype(t).itemsize) for n, (s, t) in shapes.items()}
    outs = [bufs[n] for n in ("idx", "w", "counts", "offsets", "perm_src", "inv")]
    if static:
        check(L.moe_route_static(ctypes.byref(d), lg, *outs, None), "moe_route_static")
        bits = ctypes.c_uint32(7)
        check(L.moe_route_static_status(None, ctypes.byref(bits)), "moe_route_static_status")
        if bits.value != 0:
            raise SystemExit(f"status bits {bits.value:#x}")
    else:
        n = moe.route_workspace_size(d)
        ws = dev_alloc(n)
        check(L.moe_route(ctypes.byref(d), lg, *outs, ws, n, None), "moe_route")
        check(L.moe_check_status(ws, None, None), "moe_check_status")
    res = {n: to_host(bufs[n], *shapes[n]) for n in shapes}
    return res


def compare(a, b, tag):
    for n in a:
        if not np.array_equal(a[n], b[n]):
            raise SystemExit(f"{tag}: {n} differs")


d = moe.dims(300, 128, 128, 384, 8, 1)
lg = np.random.default_rng(5).standard_normal((d.T, d.E)).astype(np.float32)
compare(route(d, lg, True), route(d, lg, False), "before reset")
check(rt.cudaDeviceReset(), "cudaDeviceReset")
lg2 = np.random.default_rng(6).standard_normal((d.T, d.E)).astype(np.float32)
compare(route(d, lg2, True), route(d, lg2, False), "after reset")
print("ok")
