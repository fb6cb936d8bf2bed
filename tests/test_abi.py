"""The C ABI without a GPU: the library builds and loads, exports exactly what include/nvfp4.h
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from conftest import ROOT

import nvfp4_block_scaled_row_gb300 as nv
from nvfp4_block_scaled_row_gb300 import build as nvbuild

HEADER = os.path.join(ROOT, "include", "nvfp4.h")
OK, INVALID, SHAPE, ALIGN, CUDA, TIMEOUT, OFFSETS, WORKSPACE = range(8)


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return nv.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_exports_match_header(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", nvbuild.LIBRARY], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(set(re.findall(r"\bT (nvfp4_[a-z0-9_]+)$", out, flags=re.M)))
    assert exported == declared_functions()
    for name in declared_functions():
        assert hasattr(lib, name)


def test_no_link_time_dependency_on_the_driver_or_a_library_gemm():
    out = subprocess.run(["ldd", nvbuild.LIBRARY], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out
    assert "cublas" not in out.lower()


def test_status_strings(lib):
    for code in range(8):
        s = nv.nvfp4_status_string(code)
        assert s and s != "unknown status"
    assert nv.nvfp4_status_string(99) == "unknown status"
    assert nv.nvfp4_abi_version() == 1
    assert nv.nvfp4_tensor_workspace_bytes() >= 4


def P(v):
    return ctypes.c_void_p(v)


def test_quantize_rowwise_host_validation(lib):
    q = lib.nvfp4_quantize_rowwise
    good = dict(x=P(1 << 20), rows=4, cols=64, off=None, g=0, mode=1, codes=P(2 << 20),
                scales=P(3 << 20), rs=P(4 << 20))

    def call(**kw):
        a = {**good, **kw}
        return q(a["x"], a["rows"], a["cols"], a["off"], a["g"], a["mode"], a["codes"],
                 a["scales"], a["rs"], None)

    assert call(cols=24) == SHAPE
    assert call(cols=0) == SHAPE
    assert call(cols=65536 + 16) == SHAPE
    assert call(mode=3) == INVALID
    assert call(rows=-1) == INVALID
    assert call(rows=0, x=None, codes=None, scales=None, rs=None) == OK  # empty: no-op
    assert call(x=None) == INVALID
    assert call(rs=None) == INVALID
    assert call(x=P((1 << 20) + 8)) == ALIGN
    assert call(codes=P((2 << 20) + 4)) == ALIGN
    assert call(rs=P((4 << 20) + 2)) == ALIGN
    assert call(codes=P((1 << 20) + 64)) == INVALID  # overlaps x
    assert call(g=3) == INVALID                       # groups without offsets
    assert call(off=P(5 << 20), g=-1) == INVALID


def test_tensor_and_fused_host_validation(lib):
    ws_bytes = nv.nvfp4_tensor_workspace_bytes()
    args = (P(1 << 20), 4, 64, 1, P(2 << 20), P(3 << 20), P(4 << 20))
    assert lib.nvfp4_quantize_tensor(*args, None, ws_bytes, None) == WORKSPACE
    assert lib.nvfp4_quantize_tensor(*args, P(5 << 20), ws_bytes - 4, None) == WORKSPACE
    assert lib.nvfp4_quantize_tensor(*args, P((5 << 20) + 4), ws_bytes, None) == WORKSPACE
    f = lib.nvfp4_fused_roundtrip
    assert f(P(1 << 20), 4, 64, 7, 1, P(2 << 20), P(3 << 20), P(4 << 20), P(6 << 20), None, 0,
             None) == INVALID
    assert f(P(1 << 20), 4, 64, 0, 1, P(2 << 20), P(3 << 20), P(4 << 20), None, None, 0,
             None) == INVALID  # y missing
    assert f(P(1 << 20), 4, 64, 0, 1, P(2 << 20), P(3 << 20), P(4 << 20), P((6 << 20) + 2),
             None, 0, None) == ALIGN
    assert f(P(1 << 20), 4, 64, 1, 1, P(2 << 20), P(3 << 20), P(4 << 20), P(6 << 20), None, 0,
             None) == WORKSPACE  # tensor scale needs the workspace
    assert lib.nvfp4_tensor_amax(P(1 << 20), -1, P(2 << 20), P(3 << 20), ws_bytes, None) == INVALID
    assert lib.nvfp4_quantize_tensor_with_amax(*args[:4], None, *args[4:], None) == INVALID


def test_dequantize_host_validation(lib):
    d = lib.nvfp4_dequantize
    args = dict(c=P(1 << 20), s=P(2 << 20), sc=P(3 << 20), k=0, rows=4, cols=64, y=P(4 << 20))

    def call(**kw):
        a = {**args, **kw}
        return d(a["c"], a["s"], a["sc"], a["k"], a["rows"], a["cols"], a["y"], None)

    assert call(k=2) == INVALID
    assert call(cols=40) == SHAPE
    assert call(rows=0, c=None, s=None, sc=None, y=None) == OK
    assert call(y=P((4 << 20) + 8)) == ALIGN
    assert call(c=P((1 << 20) + 2)) == ALIGN
    assert call(y=P((1 << 20) + 16)) == INVALID  # y overlaps the codes


def test_swizzle_and_gemm_host_validation(lib):
    sw = lib.nvfp4_swizzle_block_scales
    assert sw(P(1 << 20), -1, 64, P(2 << 20), None) == INVALID
    assert sw(P(1 << 20), 4, 40, P(2 << 20), None) == SHAPE
    assert sw(None, 0, 64, None, None) == OK
    assert sw(P(1 << 20), 4, 64, P((2 << 20) + 8), None) == ALIGN  # 16-byte lines
    assert sw(P(1 << 20), 4, 64, P(1 << 20), None) == INVALID  # overlaps the input
    g = lib.nvfp4_gemm_nt
    assert lib.nvfp4_gemm_workspace_bytes(256, 256) == 0  # no scratch memory
    ok = [P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), P(6 << 20)]
    assert g(*ok, 256, 256, 96, P(7 << 20), None, 0, None) == SHAPE  # k % 64
    assert g(*ok, 256, 250, 128, P(7 << 20), None, 0, None) == SHAPE  # n % 16
    assert g(*ok, -1, 256, 128, P(7 << 20), None, 0, None) == INVALID
    assert g(*ok, 0, 256, 128, P(7 << 20), None, 0, None) == OK
    assert g(*ok, 256, 256, 128, P((7 << 20) + 8), None, 0, None) == ALIGN  # y
    bad_scale = [ok[0], ok[1], P((3 << 20) + 2)] + ok[3:]
    assert g(*bad_scale, 256, 256, 128, P(7 << 20), None, 0, None) == ALIGN  # row scale
    bad_codes = [P((1 << 20) + 128)] + ok[1:]
    assert g(*bad_codes, 256, 256, 128, P(7 << 20), None, 0, None) == ALIGN  # TMA base


def test_launch_config_validation(lib):
    assert lib.nvfp4_set_launch_config(-1, 0, 0) == INVALID
    assert lib.nvfp4_set_launch_config(0, 99, 0) == INVALID
    assert lib.nvfp4_set_launch_config(17, 0, 0) == INVALID
    assert lib.nvfp4_set_launch_config(0, 5, 0) == INVALID
    assert lib.nvfp4_set_launch_config(2, 2, 5) == OK
    assert lib.nvfp4_set_launch_config(0, 0, 0) == OK


def test_binding_rejects_host_tensors(lib):
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        nv.nvfp4_quantize_rowwise(x)
    with pytest.raises(ValueError):
        nv.nvfp4_fused_roundtrip(x)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(nv, "_lib", None)
    monkeypatch.setattr(nv._build, "LIBRARY", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        nv.library()


def test_host_roundtrip_validation(lib):
    f = lib.nvfp4_fused_roundtrip_host
    ws = nv.nvfp4_roundtrip_host_workspace_bytes(7168)
    assert ws > 0 and nv.nvfp4_roundtrip_host_workspace_bytes(24) == 0
    args = [P(1 << 20), 4, 7168, 1, P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20)]
    assert f(*args, P(6 << 20), ws - 1, None) == WORKSPACE
    assert f(*args, P((6 << 20) + 16), ws, None) == WORKSPACE
    assert f(P(1 << 20), 4, 24, 1, P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), P(6 << 20),
             ws, None) == SHAPE
    assert f(P(1 << 20), 0, 7168, 1, None, None, None, None, None, 0, None) == OK
    assert f(None, 4, 7168, 1, P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), P(6 << 20), ws,
             None) == INVALID


def test_withhold_row_hook_validation(lib):
    h = lib.nvfp4_selftest_withhold_row
    assert h(-2, 1000) == INVALID
    assert h(3, 0) == INVALID
    assert h(3, 4_000_000_001) == INVALID
    assert h(-1, 0) == OK  # normal operation
