"""Host-side checks of the C interface (no GPU needed): every symbol declared in
include/moe.h is exported by libmoe.so, and argument / shape validation rejects bad
calls before anything is launched."""

import ctypes
import os
import re

import pytest

import moe_expert_ffn_scan_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        from moe_expert_ffn_scan_gb300 import build
        build.build()
    return moe.lib()


def test_header_declares_the_hot_path(lib):
    names = _declared_functions()
    for n in ("moe_route", "moe_quant_act", "moe_grouped_gemm_w13", "moe_swiglu_quant",
              "moe_grouped_gemm_w2", "moe_combine", "moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), f"libmoe.so does not export {n}"


def test_error_strings(lib):
    for code in range(6):
        assert lib.moe_error_string(code)
    assert b"unknown" in lib.moe_error_string(99)


def test_workspace_sizes_and_unsupported_shapes(lib):
    ok = moe.dims(7, 7168, 3072, 384, 8, 1)
    assert moe.workspace_size(ok) > moe.gemm_workspace_size(ok) > 0
    assert moe.route_workspace_size(ok) > 0
    for bad in (moe.dims(7, 7100, 3072, 384, 8, 1),   # H % 128
                moe.dims(7, 7168, 3000, 384, 8, 1),   # I % 128
                moe.dims(0, 512, 256, 8, 2, 0),       # T
                moe.dims(4, 512, 256, 8, 9, 0),       # k > E
                moe.dims(4, 512, 256, 2000, 8, 0),    # E > 1024
                moe.dims(4, 512, 256, 64, 17, 0),     # k > 16
                moe.dims(4, 512, 256, 8, 2, 2)):      # has_shared not 0/1
        assert moe.workspace_size(bad) == 0


def test_validation_happens_before_any_launch(lib):
    d = moe.dims(7, 512, 256, 8, 2, 0)
    P = ctypes.c_void_p
    # null pointers -> invalid argument, unsupported dims -> unsupported shape
    assert lib.moe_route(ctypes.byref(d), None, None, None, None, None, None, None, None, 0,
                         None) == 1
    bad = moe.dims(7, 500, 256, 8, 2, 0)
    assert lib.moe_forward(ctypes.byref(bad), None, None, None, None, None, None, 0, None) == 2
    assert lib.moe_quant_act(4, 100, None, None, None, None) == 2
    assert lib.moe_quant_act(0, 128, None, None, None, None) == 0
    assert lib.moe_swiglu_quant(4, 100, None, None, None, None) == 2
    # misaligned workspace -> invalid argument
    fake = P(0x1000 + 8)
    assert lib.moe_route(ctypes.byref(d), P(0x1000), P(0x1000), P(0x1000), P(0x1000),
                         P(0x1000), P(0x1000), P(0x1000), fake, 1 << 20, None) == 1
    # misaligned logits or outputs -> invalid argument
    for i in range(7):
        ptrs = [P(0x1000)] * 7
        ptrs[i] = P(0x1002)
        assert lib.moe_route(ctypes.byref(d), *ptrs, P(0x10000), 1 << 20, None) == 1
        lib.moe_route_static.argtypes = [ctypes.POINTER(moe.moe_dims)] + [P] * 8
        assert lib.moe_route_static(ctypes.byref(d), *ptrs, None) == 1
    # workspace too small
    assert lib.moe_route(ctypes.byref(d), P(0x1000), P(0x1000), P(0x1000), P(0x1000),
                         P(0x1000), P(0x1000), P(0x1000), P(0x10000), 16, None) == 3
    assert lib.moe_selftest_wait_timeout(None, None) == 1
    assert lib.moe_selftest_wait_timeout(P(0x1008), None) == 1
    # host-buffer forward: dims, nulls, workspace size and alignment
    w = moe.moe_weights(0x10000, 0x10000, 0x10000, 0x10000)
    assert lib.moe_forward_host(ctypes.byref(bad), P(0x1000), P(0x1000), ctypes.byref(w),
                                P(0x1000), P(0x10000), 1 << 30, None) == 2
    assert lib.moe_forward_host(ctypes.byref(d), None, P(0x1000), ctypes.byref(w), P(0x1000),
                                P(0x10000), 1 << 30, None) == 1
    assert lib.moe_forward_host(ctypes.byref(d), P(0x1000), P(0x1000), ctypes.byref(w),
                                P(0x1000), P(0x10000), 16, None) == 3
    assert lib.moe_forward_host(ctypes.byref(d), P(0x1000), P(0x1000), ctypes.byref(w),
                                P(0x1000), P(0x10008), 1 << 30, None) == 1
    assert moe.host_workspace_size(d) > moe.workspace_size(d)
    # host-buffer pipeline: sizes, then checks before any stream or event is created
    assert moe.host_pipeline_workspace_size(d, 1) == moe.host_workspace_size(d)
    assert moe.host_pipeline_workspace_size(d, 2) > moe.host_pipeline_workspace_size(d, 1)
    assert moe.host_pipeline_workspace_size(d, 0) == 0
    assert moe.host_pipeline_workspace_size(d, 9) == 0
    assert moe.host_pipeline_workspace_size(bad, 2) == 0
    h = P()
    big = moe.host_pipeline_workspace_size(d, 2)
    assert lib.moe_host_pipeline_create(ctypes.byref(d), ctypes.byref(w), 2, P(0x10000), big,
                                        None) == 1
    assert lib.moe_host_pipeline_create(ctypes.byref(bad), ctypes.byref(w), 2, P(0x10000), big,
                                        ctypes.byref(h)) == 2
    for depth in (0, 9):
        assert lib.moe_host_pipeline_create(ctypes.byref(d), ctypes.byref(w), depth,
                                            P(0x10000), big, ctypes.byref(h)) == 1
    assert lib.moe_host_pipeline_create(ctypes.byref(d), None, 2, P(0x10000), big,
                                        ctypes.byref(h)) == 1
    assert lib.moe_host_pipeline_create(ctypes.byref(d), ctypes.byref(w), 2, P(0x10008), big,
                                        ctypes.byref(h)) == 1
    assert lib.moe_host_pipeline_create(ctypes.byref(d), ctypes.byref(w), 2, P(0x10000),
                                        big - 1, ctypes.byref(h)) == 3
    assert h.value is None  # nothing was created
    assert lib.moe_host_pipeline_submit(None, P(0x1000), P(0x1000), P(0x1000)) == 1
    assert lib.moe_host_pipeline_sync(None) == 1
    assert lib.moe_host_pipeline_destroy(None) == 1
    # router projection: shape checks, then null / misaligned pointers
    assert lib.moe_router_logits(0, 128, 8, P(0x1000), P(0x1000), P(0x1000), None) == 2
    assert lib.moe_router_logits(4, 120, 8, P(0x1000), P(0x1000), P(0x1000), None) == 2
    assert lib.moe_router_logits(4, 128, 0, P(0x1000), P(0x1000), P(0x1000), None) == 2
    assert lib.moe_router_logits(4, 128, 8, None, P(0x1000), P(0x1000), None) == 1
    assert lib.moe_router_logits(4, 128, 8, P(0x1008), P(0x1000), P(0x1000), None) == 1
    assert lib.moe_router_logits(4, 128, 8, P(0x1000), P(0x1004), P(0x1000), None) == 1
    w = moe.moe_weights(0x10000, 0x10000, 0x10008, 0x10000)  # w2 misaligned (needs 32 B)
    assert lib.moe_forward(ctypes.byref(d), P(0x1000), P(0x1000), ctypes.byref(w),
                           P(0x1000), None, P(0x10000), 1 << 30, None) == 1


def test_forward_options_validated_before_any_launch(lib):
    """moe_forward_ex: option values outside {0, 1}, and chunk sizes that are not a
    multiple of 16 in [144, 224], are rejected before anything launches; a valid option
    set gets as far as the workspace-size check."""
    d = moe.dims(7, 512, 256, 8, 2, 0)
    W = moe.moe_weights(0x10000, 0x10000, 0x10000, 0x10000)
    P = ctypes.c_void_p

    def call(opt, ws_bytes=1 << 30):
        return lib.moe_forward_ex(ctypes.byref(d), P(0x1000), P(0x1000), ctypes.byref(W),
                                  ctypes.byref(opt), P(0x1000), None, None, P(0x10000),
                                  ws_bytes, None)
    for bad in ((2, 0, 0, 0), (0, 2, 0, 0), (0, 0, 2, 0), (0, 0, 0, 100), (0, 0, 0, 150),
                (0, 0, 0, 240), (0, 0, 0, 128), (0, 0, 0, -16)):
        assert call(moe.moe_options(*bad)) == 1, bad
    for ok in ((0, 0, 0, 0), (0, 0, 0, 144), (0, 0, 0, 176), (0, 0, 0, 224), (1, 0, 1, 160)):
        assert call(moe.moe_options(*ok), ws_bytes=16) == 3, ok


def test_nvfp4_validation_before_any_launch(lib):
    P = ctypes.c_void_p
    ok = moe.dims(7, 7168, 3072, 384, 8, 1)
    assert moe.workspace_size_nvfp4(ok) > moe.gemm_workspace_size_nvfp4(ok) > 0
    # the NVFP4 GEMMs need H and I multiples of 256 (their scale rows are whole TMA rows)
    for bad in (moe.dims(7, 7168 + 128, 3072, 384, 8, 1), moe.dims(7, 7168, 3072 - 128, 384, 8, 1)):
        assert moe.workspace_size(bad) > 0 and moe.workspace_size_nvfp4(bad) == 0
        assert lib.moe_forward_nvfp4(ctypes.byref(bad), P(0x1000), P(0x1000), None, P(0x1000),
                                     None, P(0x10000), 1 << 30, None) == 2
        assert lib.moe_grouped_gemm_w13_nvfp4(ctypes.byref(bad), *[P(0x1000)] * 8, P(0x10000),
                                              1 << 30, None) == 2
    d = moe.dims(7, 512, 256, 8, 2, 0)
    assert lib.moe_forward_nvfp4(ctypes.byref(d), P(0x1000), P(0x1000), None, P(0x1000), None,
                                 P(0x10000), 1 << 30, None) == 1
    w = moe.moe_weights_nvfp4(0x10000, 0x10000, 0x10002, 0x10000, 0x10000, None)  # gs misaligned
    assert lib.moe_forward_nvfp4(ctypes.byref(d), P(0x1000), P(0x1000), ctypes.byref(w),
                                 P(0x1000), None, P(0x10000), 1 << 30, None) == 1
    w = moe.moe_weights_nvfp4(0x10000, 0x10000, None, 0x10000, 0x10000, None)
    assert lib.moe_forward_nvfp4(ctypes.byref(d), P(0x1000), P(0x1000), ctypes.byref(w),
                                 P(0x1000), None, P(0x10000), 16, None) == 3
    assert lib.moe_grouped_gemm_w2_nvfp4(ctypes.byref(d), None, *[P(0x1000)] * 6, P(0x10000),
                                         1 << 30, None) == 1
    assert lib.moe_grouped_gemm_w2_nvfp4(ctypes.byref(d), *[P(0x1000)] * 7, P(0x10000), 16,
                                         None) == 3


def test_router_split_validation(lib):
    P = ctypes.c_void_p
    assert moe.lib().moe_router_split_bytes(384, 7168) == 3 * 384 * 7168 * 2
    assert moe.lib().moe_router_split_bytes(8, 100) == 0
    assert lib.moe_router_split(8, 100, P(0x1000), P(0x1000), None) == 2
    assert lib.moe_router_split(8, 128, P(0x1000), P(0x1008), None) == 1
    assert lib.moe_router_logits_split(0, 128, 8, P(0x1000), P(0x1000), P(0x1000), None) == 2
    assert lib.moe_router_logits_split(4, 128, 8, P(0x1008), P(0x1000), P(0x1000), None) == 1
    assert lib.moe_router_logits_split(4, 128, 8, P(0x1000), None, P(0x1000), None) == 1


def test_python_binding_rejects_host_tensors(lib):
    import torch
    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        moe.moe_quant_act(x, torch.zeros(4, 128, dtype=torch.uint8),
                          torch.zeros(4, 1, dtype=torch.uint8))


def test_missing_library_fails_loudly(monkeypatch):
    """No fallback: with the library absent every call raises instead of computing
    anything another way."""
    monkeypatch.setattr(moe, "_LIB", None)
    monkeypatch.setattr(moe, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmoe.so"))
    with pytest.raises(RuntimeError, match="missing"):
        moe.workspace_size(moe.dims(7, 512, 256, 8, 2, 0))
    with pytest.raises(RuntimeError, match="missing"):
        moe.MoELayer(512, 256, 8, 2, 0, None, None, None, None).workspace(7)


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/moe.h compiles as pedantic C99 and a C program links against libmoe.so
    and queries a workspace size (host-only call)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "t.c"
    src.write_text(
        '#include "moe.h"\n#include <stdio.h>\n'
        'int main(void) { moe_dims d = {7, 7168, 3072, 384, 8, 1};\n'
        '  printf("%zu\\n", moe_workspace_size(&d)); return 0; }\n')
    exe = tmp_path / "t"
    libdir = os.path.dirname(moe.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I" + os.path.join(ROOT, "include"), str(src), "-L" + libdir, "-lmoe",
                        "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    assert int(out) == moe.workspace_size(moe.dims(7, 7168, 3072, 384, 8, 1)) > 0
