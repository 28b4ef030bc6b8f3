"""Python binding of libmoe.so, the GB300 routed-MoE expert FFN (MXFP4 weights,
online FP8 activations).

Argument marshalling only: every step runs in the library's CUDA kernels.  PyTorch
provides device memory and the current stream.  The functions carry the C names
(see include/moe.h for argument meaning, layouts and errors); each raises
MoeError when the C call returns a non-zero status.  Importing this package does
not need a GPU; calling into the library does, and fails loudly if libmoe.so has
not been built (python -m moe_expert_ffn_scan_gb300.build).
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
STATUS_WAIT_TIMEOUT = 1
STATUS_BAD_INDEX = 2
STATUS_BAD_PLAN = 4


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        msg = lib().moe_error_string(code).decode() if _LIB is not None else str(code)
        super().__init__(f"{fn}: status {code} ({msg})")
        self.code = code


class moe_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "I", "E", "k", "has_shared")]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w13", "w13_s", "w2", "w2_s")]


class moe_options(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("fuse_combine", "fuse_swiglu", "pair_tiles",
                                              "large_chunk_rows")]


class moe_weights_nvfp4(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w13", "w13_s", "w13_gs", "w2", "w2_s", "w2_gs")]


DEBUG_FIELDS = ("idx", "w", "counts", "offsets", "perm_src", "inv", "xq", "xs", "y13", "hq",
                "hs", "y2")


class moe_debug_out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in DEBUG_FIELDS]


_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t
_DP = ctypes.POINTER(moe_dims)


def lib():
    """Load libmoe.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m moe_expert_ffn_scan_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.moe_error_string.argtypes = [ctypes.c_int]
        L.moe_error_string.restype = ctypes.c_char_p
        for fn in ("moe_workspace_size", "moe_route_workspace_size", "moe_gemm_workspace_size",
                   "moe_host_workspace_size", "moe_workspace_size_nvfp4",
                   "moe_gemm_workspace_size_nvfp4"):
            getattr(L, fn).argtypes = [_DP]
            getattr(L, fn).restype = _SZ
        L.moe_route.argtypes = [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
        L.moe_quant_act.argtypes = [_I, _I, _P, _P, _P, _P]
        L.moe_router_split_bytes.argtypes = [_I, _I]
        L.moe_router_split_bytes.restype = _SZ
        L.moe_router_split.argtypes = [_I, _I, _P, _P, _P]
        L.moe_router_split.restype = ctypes.c_int
        L.moe_router_logits_split.argtypes = [_I, _I, _I, _P, _P, _P, _P]
        L.moe_router_logits_split.restype = ctypes.c_int
        L.moe_router_logits.argtypes = [_I, _I, _I, _P, _P, _P, _P]
        L.moe_grouped_gemm_w13.argtypes = [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
        L.moe_swiglu_quant.argtypes = [_I, _I, _P, _P, _P, _P]
        L.moe_grouped_gemm_w2.argtypes = [_DP, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
        L.moe_combine.argtypes = [_DP, _P, _P, _P, _P, _P]
        L.moe_forward.argtypes = [_DP, _P, _P, ctypes.POINTER(moe_weights), _P,
                                  ctypes.POINTER(moe_debug_out), _P, _SZ, _P]
        L.moe_forward_host.argtypes = [_DP, _P, _P, ctypes.POINTER(moe_weights), _P, _P, _SZ,
                                       _P]
        L.moe_forward_timed.argtypes = [_DP, _P, _P, ctypes.POINTER(moe_weights), _P,
                                        ctypes.POINTER(moe_debug_out), ctypes.POINTER(_P), _P,
                                        _SZ, _P]
        _WN = ctypes.POINTER(moe_weights_nvfp4)
        L.moe_forward_nvfp4.argtypes = [_DP, _P, _P, _WN, _P, ctypes.POINTER(moe_debug_out), _P,
                                        _SZ, _P]
        L.moe_forward_nvfp4_timed.argtypes = [_DP, _P, _P, _WN, _P,
                                              ctypes.POINTER(moe_debug_out), ctypes.POINTER(_P),
                                              _P, _SZ, _P]
        L.moe_grouped_gemm_w13_nvfp4.argtypes = [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                                 _P]
        L.moe_grouped_gemm_w2_nvfp4.argtypes = [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
        L.moe_forward_ex.argtypes = [_DP, _P, _P, ctypes.POINTER(moe_weights),
                                     ctypes.POINTER(moe_options), _P,
                                     ctypes.POINTER(moe_debug_out), ctypes.POINTER(_P), _P, _SZ,
                                     _P]
        L.moe_route_static.argtypes = [_DP, _P, _P, _P, _P, _P, _P, _P, _P]
        L.moe_route_static_status.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32)]
        L.moe_check_status.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_uint32)]
        L.moe_selftest_wait_timeout.argtypes = [_P, _P]
        L.moe_host_pipeline_workspace_size.argtypes = [_DP, _I]
        L.moe_host_pipeline_workspace_size.restype = _SZ
        L.moe_host_pipeline_create.argtypes = [_DP, ctypes.POINTER(moe_weights), _I, _P, _SZ,
                                               ctypes.POINTER(_P)]
        L.moe_host_pipeline_submit.argtypes = [_P, _P, _P, _P]
        L.moe_host_pipeline_sync.argtypes = [_P]
        L.moe_host_pipeline_destroy.argtypes = [_P]
        for fn in ("moe_host_pipeline_create", "moe_host_pipeline_submit",
                   "moe_host_pipeline_sync", "moe_host_pipeline_destroy"):
            getattr(L, fn).restype = ctypes.c_int
        for fn in ("moe_route", "moe_quant_act", "moe_grouped_gemm_w13", "moe_swiglu_quant",
                   "moe_grouped_gemm_w2", "moe_combine", "moe_forward", "moe_forward_timed",
                   "moe_check_status", "moe_forward_nvfp4", "moe_forward_nvfp4_timed",
                   "moe_grouped_gemm_w13_nvfp4", "moe_grouped_gemm_w2_nvfp4",
                   "moe_route_static", "moe_route_static_status", "moe_forward_ex"):
            getattr(L, fn).restype = ctypes.c_int
        _LIB = L
    return _LIB


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if t.device.type != "cuda":
        raise ValueError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def dims(T, H, I, E, k, has_shared):
    return moe_dims(int(T), int(H), int(I), int(E), int(k), int(has_shared))


def _d(d):
    if not isinstance(d, moe_dims):
        d = dims(d.T, d.H, d.I, d.E, d.k, d.has_shared)
    return ctypes.byref(d)


def workspace_size(d) -> int:
    return lib().moe_workspace_size(_d(d))


def host_workspace_size(d) -> int:
    return lib().moe_host_workspace_size(_d(d))


def host_pipeline_workspace_size(d, depth) -> int:
    return lib().moe_host_pipeline_workspace_size(_d(d), depth)


def workspace_size_nvfp4(d) -> int:
    return lib().moe_workspace_size_nvfp4(_d(d))


def gemm_workspace_size_nvfp4(d) -> int:
    return lib().moe_gemm_workspace_size_nvfp4(_d(d))


def route_workspace_size(d) -> int:
    return lib().moe_route_workspace_size(_d(d))


def gemm_workspace_size(d) -> int:
    return lib().moe_gemm_workspace_size(_d(d))


def alloc_workspace(nbytes, device="cuda"):
    """A workspace tensor (torch allocations are 256-byte aligned or better)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def moe_route(d, logits, idx, w, counts, offsets, perm_src, inv, ws, stream=None):
    _check("moe_route", lib().moe_route(_d(d), _p(logits), _p(idx), _p(w), _p(counts),
                                        _p(offsets), _p(perm_src), _p(inv), _p(ws),
                                        ws.numel(), _stream(stream)))


def moe_router_logits(x, wg, logits, stream=None):
    """logits [T, E] fp32 = x [T, H] bf16 . wg [E, H] fp32 ^T (router gate projection)."""
    T, H = x.shape
    E = wg.shape[0]
    _check("moe_router_logits", lib().moe_router_logits(T, H, E, _p(x), _p(wg), _p(logits),
                                                        _stream(stream)))


def moe_router_split(wg, wg3=None, stream=None):
    """Splits the fp32 gate weight [E, H] into the three bf16 pieces [3, E, H] the
    tensor-core router projection reads (hi + mid + lo == wg).  Returns wg3."""
    E, H = wg.shape
    if wg3 is None:
        wg3 = torch.empty(3, E, H, dtype=torch.bfloat16, device=wg.device)
    _check("moe_router_split", lib().moe_router_split(E, H, _p(wg), _p(wg3), _stream(stream)))
    return wg3


def moe_router_logits_split(x, wg3, logits, stream=None):
    """logits [T, E] fp32 = x [T, H] bf16 . wg^T on the tensor cores, from the pieces of
    moe_router_split."""
    T, H = x.shape
    E = wg3.shape[1]
    _check("moe_router_logits_split", lib().moe_router_logits_split(
        T, H, E, _p(x), _p(wg3), _p(logits), _stream(stream)))


def moe_quant_act(x, q, s, stream=None):
    rows, cols = x.shape
    _check("moe_quant_act", lib().moe_quant_act(rows, cols, _p(x), _p(q), _p(s),
                                                _stream(stream)))


def moe_grouped_gemm_w13(d, xq, xs, perm_src, group_offsets, w13, w13_s, y13, ws, stream=None):
    _check("moe_grouped_gemm_w13", lib().moe_grouped_gemm_w13(
        _d(d), _p(xq), _p(xs), _p(perm_src), _p(group_offsets), _p(w13), _p(w13_s), _p(y13),
        _p(ws), ws.numel(), _stream(stream)))


def moe_swiglu_quant(y13, hq, hs, stream=None):
    rows, two_i = y13.shape
    _check("moe_swiglu_quant", lib().moe_swiglu_quant(rows, two_i // 2, _p(y13), _p(hq), _p(hs),
                                                      _stream(stream)))


def moe_grouped_gemm_w2(d, hq, hs, group_offsets, w2, w2_s, y2, ws, stream=None):
    _check("moe_grouped_gemm_w2", lib().moe_grouped_gemm_w2(
        _d(d), _p(hq), _p(hs), _p(group_offsets), _p(w2), _p(w2_s), _p(y2), _p(ws),
        ws.numel(), _stream(stream)))


def moe_combine(d, y2, inv, w, out, stream=None):
    _check("moe_combine", lib().moe_combine(_d(d), _p(y2), _p(inv), _p(w), _p(out),
                                            _stream(stream)))


def moe_forward(d, x, logits, w13, w13_s, w2, w2_s, out, ws, debug=None, stream=None):
    W = moe_weights(_p(w13), _p(w13_s), _p(w2), _p(w2_s))
    dbg = None
    if debug:
        dbg = moe_debug_out(*[_p(debug.get(n)) for n in DEBUG_FIELDS])
    _check("moe_forward", lib().moe_forward(
        _d(d), _p(x), _p(logits), ctypes.byref(W), _p(out),
        ctypes.byref(dbg) if dbg is not None else None, _p(ws), ws.numel(), _stream(stream)))


def _nv_weights(w13, w13_s, w13_gs, w2, w2_s, w2_gs):
    return moe_weights_nvfp4(_p(w13), _p(w13_s), _p(w13_gs), _p(w2), _p(w2_s), _p(w2_gs))


def moe_forward_nvfp4(d, x, logits, w13, w13_s, w13_gs, w2, w2_s, w2_gs, out, ws, debug=None,
                      stream=None):
    """moe_forward with NVFP4 expert weights (codes, E4M3 scales per 16, fp32 tensor
    scales [G, 2] / [G] or None); ws: workspace_size_nvfp4(d) bytes."""
    W = _nv_weights(w13, w13_s, w13_gs, w2, w2_s, w2_gs)
    dbg = None
    if debug:
        dbg = moe_debug_out(*[_p(debug.get(n)) for n in DEBUG_FIELDS])
    _check("moe_forward_nvfp4", lib().moe_forward_nvfp4(
        _d(d), _p(x), _p(logits), ctypes.byref(W), _p(out),
        ctypes.byref(dbg) if dbg is not None else None, _p(ws), ws.numel(), _stream(stream)))


def moe_forward_nvfp4_timed(d, x, logits, w13, w13_s, w13_gs, w2, w2_s, w2_gs, out, ws, events,
                            stream=None):
    W = _nv_weights(w13, w13_s, w13_gs, w2, w2_s, w2_gs)
    ev = (_P * 8)(*[e.cuda_event for e in events])
    _check("moe_forward_nvfp4_timed", lib().moe_forward_nvfp4_timed(
        _d(d), _p(x), _p(logits), ctypes.byref(W), _p(out), None, ev, _p(ws), ws.numel(),
        _stream(stream)))


def moe_grouped_gemm_w13_nvfp4(d, xq, xs, perm_src, group_offsets, w13, w13_s, w13_gs, y13, ws,
                               stream=None):
    _check("moe_grouped_gemm_w13_nvfp4", lib().moe_grouped_gemm_w13_nvfp4(
        _d(d), _p(xq), _p(xs), _p(perm_src), _p(group_offsets), _p(w13), _p(w13_s), _p(w13_gs),
        _p(y13), _p(ws), ws.numel(), _stream(stream)))


def moe_grouped_gemm_w2_nvfp4(d, hq, hs, group_offsets, w2, w2_s, w2_gs, y2, ws, stream=None):
    _check("moe_grouped_gemm_w2_nvfp4", lib().moe_grouped_gemm_w2_nvfp4(
        _d(d), _p(hq), _p(hs), _p(group_offsets), _p(w2), _p(w2_s), _p(w2_gs), _p(y2), _p(ws),
        ws.numel(), _stream(stream)))


def moe_route_static(d, logits, idx, w, counts, offsets, perm_src, inv, stream=None):
    """moe_route without a workspace: its scratch is a fixed array inside the library
    (calls must not overlap on the GPU)."""
    _check("moe_route_static", lib().moe_route_static(
        _d(d), _p(logits), _p(idx), _p(w), _p(counts), _p(offsets), _p(perm_src), _p(inv),
        _stream(stream)))


def moe_route_static_status(stream=None) -> int:
    """Synchronises the stream and returns the device status bits of moe_route_static's
    fixed array (those of its last call)."""
    bits = ctypes.c_uint32(0)
    rc = lib().moe_route_static_status(_stream(stream), ctypes.byref(bits))
    if rc not in (MOE_OK, 5):
        raise MoeError("moe_route_static_status", rc)
    return bits.value


def moe_forward_ex(d, x, logits, w13, w13_s, w2, w2_s, out, ws, fuse_combine=False,
                   fuse_swiglu=False, pair_tiles=False, large_chunk_rows=0, debug=None,
                   events=None, stream=None):
    """moe_forward with options (fuse_combine: the W2 GEMM's epilogue performs the
    weighted top-k combine + shared add; fuse_swiglu: the W13 GEMM's epilogue performs
    SwiGLU + FP8 quantisation; pair_tiles: groups above 64 rows on SM pairs;
    large_chunk_rows: the tile plan's chunk size for groups above 64 rows, 0 = 224) and
    optional stage events."""
    W = moe_weights(_p(w13), _p(w13_s), _p(w2), _p(w2_s))
    opt = moe_options(int(bool(fuse_combine)), int(bool(fuse_swiglu)), int(bool(pair_tiles)),
                      int(large_chunk_rows))
    dbg = None
    if debug:
        dbg = moe_debug_out(*[_p(debug.get(n)) for n in DEBUG_FIELDS])
    ev = (_P * 8)(*[e.cuda_event for e in events]) if events else None
    _check("moe_forward_ex", lib().moe_forward_ex(
        _d(d), _p(x), _p(logits), ctypes.byref(W), ctypes.byref(opt), _p(out),
        ctypes.byref(dbg) if dbg is not None else None, ev, _p(ws), ws.numel(),
        _stream(stream)))


def _host_p(t):
    if t.device.type != "cpu":
        raise ValueError("tensor must live in host memory")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def moe_forward_host(d, x_host, logits_host, w13, w13_s, w2, w2_s, out_host, ws, stream=None):
    """The layer from host buffers to a host buffer (two copies in, one out, on the
    stream; pinned buffers keep them asynchronous).  ws: host_workspace_size(d)."""
    W = moe_weights(_p(w13), _p(w13_s), _p(w2), _p(w2_s))
    _check("moe_forward_host", lib().moe_forward_host(
        _d(d), _host_p(x_host), _host_p(logits_host), ctypes.byref(W), _host_p(out_host),
        _p(ws), ws.numel(), _stream(stream)))


STAGES = ("route", "quant", "plan_gather", "gemm_w13", "swiglu_quant", "gemm_w2", "combine")


def moe_forward_timed(d, x, logits, w13, w13_s, w2, w2_s, out, ws, events, debug=None,
                      stream=None):
    """moe_forward recording 8 torch.cuda.Event objects at the stage boundaries (see
    STAGES); the events must already exist (recorded once)."""
    W = moe_weights(_p(w13), _p(w13_s), _p(w2), _p(w2_s))
    dbg = None
    if debug:
        dbg = moe_debug_out(*[_p(debug.get(n)) for n in DEBUG_FIELDS])
    ev = (_P * 8)(*[e.cuda_event for e in events])
    _check("moe_forward_timed", lib().moe_forward_timed(
        _d(d), _p(x), _p(logits), ctypes.byref(W), _p(out),
        ctypes.byref(dbg) if dbg is not None else None, ev, _p(ws), ws.numel(),
        _stream(stream)))


def moe_check_status(ws, stream=None) -> int:
    """Synchronises the stream and returns the device status bits of a workspace."""
    bits = ctypes.c_uint32(0)
    rc = lib().moe_check_status(_p(ws), _stream(stream), ctypes.byref(bits))
    if rc not in (MOE_OK, 5):
        raise MoeError("moe_check_status", rc)
    return bits.value


def moe_selftest_wait_timeout(ws, stream=None):
    """Runs the failure-path self-test (a wait that must time out) on ws's status word."""
    _check("moe_selftest_wait_timeout", lib().moe_selftest_wait_timeout(_p(ws), _stream(stream)))


def debug_buffers(d, device="cuda"):
    """Device buffers for every intermediate moe_forward can expose."""
    T, H, I, E, k, sh = d.T, d.H, d.I, d.E, d.k, d.has_shared
    R = T * k
    Rs = R + (T if sh else 0)
    G = E + sh
    z = lambda *s, dt: torch.empty(*s, dtype=dt, device=device)
    return dict(idx=z(T, k, dt=torch.int32), w=z(T, k, dt=torch.float32),
                counts=z(E, dt=torch.int32), offsets=z(G + 1, dt=torch.int32),
                perm_src=z(max(R, 1), dt=torch.int32), inv=z(max(R, 1), dt=torch.int32),
                xq=z(T, H, dt=torch.uint8), xs=z(T, H // 128, dt=torch.uint8),
                y13=z(Rs, 2 * I, dt=torch.bfloat16), hq=z(Rs, I, dt=torch.uint8),
                hs=z(Rs, I // 128, dt=torch.uint8), y2=z(Rs, H, dt=torch.bfloat16))


class HostGraph:
    """forward_host captured once as a CUDA graph over pinned buffers x_host [T, H]
    bf16, logits_host [T, E] fp32 and out_host [T, H] bf16.  Write a step's inputs
    into x_host / logits_host, call replay(), synchronise, read out_host."""

    def __init__(self, layer, T):
        self.layer, self.T = layer, T
        self.x_host = torch.zeros(T, layer.H, dtype=torch.bfloat16).pin_memory()
        self.logits_host = torch.zeros(T, layer.E, dtype=torch.float32).pin_memory()
        self.out_host = torch.zeros(T, layer.H, dtype=torch.bfloat16).pin_memory()
        layer.host_workspace(T)  # allocated before capture
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer.forward_host(self.x_host, self.logits_host, self.out_host)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            layer.forward_host(self.x_host, self.logits_host, self.out_host)
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()
        return self.out_host


class HostPipeline:
    """The native host-buffer pipeline (moe_host_pipeline_*): submit() enqueues one
    layer step from pinned host buffers to a pinned host buffer and returns; step i's
    copies overlap steps i-1 and i+1 on the pipeline's own streams; sync() waits for
    every submitted step.  Buffers passed to submit() stay in use until sync()."""

    def __init__(self, layer, T, depth=2):
        self.T, self.H, self.E, self.depth = T, layer.H, layer.E, depth
        d = layer.dims(T)
        size = host_pipeline_workspace_size(d, depth)
        if size == 0:
            raise ValueError(f"unsupported dims or depth {depth} (1..8)")
        self.ws = alloc_workspace(size, layer.w13.device)
        self._weights = (layer.w13, layer.w13_s, layer.w2, layer.w2_s)  # kept alive
        W = moe_weights(*[_p(t) for t in self._weights])
        h = _P()
        _check("moe_host_pipeline_create", lib().moe_host_pipeline_create(
            _d(d), ctypes.byref(W), depth, _p(self.ws), self.ws.numel(), ctypes.byref(h)))
        self._h = h

    def _host(self, t, shape, dtype):
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"expected {dtype} {shape}, got {t.dtype} {tuple(t.shape)}")
        return _host_p(t)

    def submit(self, x_host, logits_host, out_host):
        if self._h is None:
            raise RuntimeError("pipeline closed")
        _check("moe_host_pipeline_submit", lib().moe_host_pipeline_submit(
            self._h, self._host(x_host, (self.T, self.H), torch.bfloat16),
            self._host(logits_host, (self.T, self.E), torch.float32),
            self._host(out_host, (self.T, self.H), torch.bfloat16)))

    def sync(self):
        _check("moe_host_pipeline_sync", lib().moe_host_pipeline_sync(self._h))

    def close(self):
        if getattr(self, "_h", None) is not None:
            h, self._h = self._h, None
            _check("moe_host_pipeline_destroy", lib().moe_host_pipeline_destroy(h))

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoELayer:
    """The user-facing layer: resident MXFP4 weights plus a reusable workspace.

    `forward(x, logits)` runs moe_forward on the current stream and returns the
    bf16 output [T, H]."""

    def __init__(self, H, I, E, k, has_shared, w13, w13_s, w2, w2_s, fmt="mxfp4", w13_gs=None,
                 w2_gs=None, fuse_combine=False, fuse_swiglu=False, pair_tiles=False,
                 large_chunk_rows=0):
        if fmt not in ("mxfp4", "nvfp4"):
            raise ValueError(f"unknown weight format {fmt!r}")
        if (fuse_combine or fuse_swiglu or pair_tiles or large_chunk_rows) and fmt != "mxfp4":
            raise ValueError("the fusion and tile options take MXFP4 weights")
        self.fuse_combine = bool(fuse_combine)
        self.fuse_swiglu = bool(fuse_swiglu)
        self.pair_tiles = bool(pair_tiles)
        self.large_chunk_rows = int(large_chunk_rows)
        self.H, self.I, self.E, self.k, self.has_shared = H, I, E, k, has_shared
        self.w13, self.w13_s, self.w2, self.w2_s = w13, w13_s, w2, w2_s
        self.fmt, self.w13_gs, self.w2_gs = fmt, w13_gs, w2_gs
        self._ws = None
        self._T = -1

    def dims(self, T):
        return dims(T, self.H, self.I, self.E, self.k, self.has_shared)

    def workspace(self, T):
        if self._ws is None or self._T < T:
            size = (workspace_size if self.fmt == "mxfp4" else workspace_size_nvfp4)(self.dims(T))
            if size == 0:
                raise ValueError(f"unsupported dims for {self.fmt} weights")
            self._ws = alloc_workspace(size, self.w13.device)
            self._T = T
        return self._ws

    def _mxfp4_only(self, what):
        if self.fmt != "mxfp4":
            raise NotImplementedError(f"{what} takes MXFP4 weights")

    def host_workspace(self, T):
        self._mxfp4_only("the host-buffer forward")
        if getattr(self, "_hws", None) is None or self._hT < T:
            self._hws = alloc_workspace(host_workspace_size(self.dims(T)), self.w13.device)
            self._hT = T
        return self._hws

    def host_pipeline(self, T, depth=2):
        """A HostPipeline for T-token steps (its own workspace and streams)."""
        self._mxfp4_only("the host-buffer pipeline")
        return HostPipeline(self, T, depth)

    def forward_host(self, x_host, logits_host, out_host, stream=None):
        """End to end from host memory: x_host [T, H] bf16 and logits_host [T, E] fp32
        (pinned) in, out_host [T, H] bf16 (pinned) written when the stream reaches it."""
        T = x_host.shape[0]
        moe_forward_host(self.dims(T), x_host, logits_host, self.w13, self.w13_s, self.w2,
                         self.w2_s, out_host, self.host_workspace(T), stream=stream)
        return out_host

    def host_graph(self, T):
        """A CUDA graph of forward_host on layer-owned pinned buffers (see HostGraph):
        one launch per step for the copies in, the layer's kernels and the copy out."""
        return HostGraph(self, T)

    def forward(self, x, logits, out=None, debug=None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=x.device)
        if self.fmt == "mxfp4":
            moe_forward_ex(self.dims(T), x, logits, self.w13, self.w13_s, self.w2, self.w2_s, out,
                           self.workspace(T), fuse_combine=self.fuse_combine,
                           fuse_swiglu=self.fuse_swiglu, pair_tiles=self.pair_tiles,
                           large_chunk_rows=self.large_chunk_rows, debug=debug, stream=stream)
        else:
            moe_forward_nvfp4(self.dims(T), x, logits, self.w13, self.w13_s, self.w13_gs,
                              self.w2, self.w2_s, self.w2_gs, out, self.workspace(T),
                              debug=debug, stream=stream)
        return out

    CHUNK_CANDIDATES = (224, 208, 192, 176, 160, 144)

    def tune_chunk_rows(self, x, logits, candidates=CHUNK_CANDIDATES, steps=10, warmup=3):
        """Exact-shape tuning of the tile plan on a recorded batch (its routing histogram
        decides the group sizes): times the layer with each candidate chunk size for
        groups above 64 rows (CUDA events, median of `steps` forwards after `warmup`),
        keeps the fastest in self.large_chunk_rows and returns (best, {candidate: ms}).
        Every candidate gives the same output bit for bit; only the tiling changes."""
        self._mxfp4_only("chunk-size tuning")
        out = torch.empty(x.shape[0], self.H, dtype=torch.bfloat16, device=x.device)
        times = {}
        keep = self.large_chunk_rows
        try:
            for c in candidates:
                self.large_chunk_rows = int(c)
                for _ in range(warmup):
                    self.forward(x, logits, out=out)
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(steps)]
                for a, b in ev:
                    a.record()
                    self.forward(x, logits, out=out)
                    b.record()
                torch.cuda.synchronize()
                ts = sorted(a.elapsed_time(b) for a, b in ev)
                times[int(c)] = ts[len(ts) // 2]
        except Exception:
            self.large_chunk_rows = keep
            raise
        best = min(times, key=times.get)
        self.large_chunk_rows = best
        return best, times

    def forward_timed(self, x, logits, out, events, stream=None):
        """forward recording the 8 stage events of moe_forward_timed (see STAGES)."""
        T = x.shape[0]
        if self.fmt == "mxfp4":
            moe_forward_ex(self.dims(T), x, logits, self.w13, self.w13_s, self.w2, self.w2_s, out,
                           self.workspace(T), fuse_combine=self.fuse_combine,
                           fuse_swiglu=self.fuse_swiglu, pair_tiles=self.pair_tiles,
                           large_chunk_rows=self.large_chunk_rows, events=events,
                           stream=stream)
        else:
            moe_forward_nvfp4_timed(self.dims(T), x, logits, self.w13, self.w13_s, self.w13_gs,
                                    self.w2, self.w2_s, self.w2_gs, out, self.workspace(T),
                                    events, stream=stream)
        return out
