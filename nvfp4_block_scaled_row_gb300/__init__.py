"""GB300 NVFP4 quantization: per-token / per-tensor FP32 scales, E4M3 block scales with
Four-Over-Six selection, packed E2M1 codes, and the exact BF16 dequantization.

This module is a thin ctypes binding over the C ABI in include/nvfp4.h (libnvfp4_gb300.so,
built in-tree by ``nvfp4_block_scaled_row_gb300.build``).  The functions carry the C names and
only marshal arguments: they check that tensors are contiguous CUDA tensors of the right dtype
and shape, allocate outputs that were not supplied (torch is used for device memory and streams
only), and raise ``Nvfp4Error`` on any non-OK status.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.
"""
import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "Nvfp4Error", "MODE_SIX", "MODE_FOUR_OVER_SIX", "SCALE_ROW", "SCALE_TENSOR",
    "nvfp4_quantize_rowwise", "nvfp4_quantize_residual", "nvfp4_row_amax", "nvfp4_quantize_guided", "nvfp4_quantize_tensor", "nvfp4_quantize_tensor_with_amax",
    "nvfp4_tensor_amax", "nvfp4_quantize_tensor_noalloc", "nvfp4_dequantize", "nvfp4_fused_roundtrip",
    "nvfp4_swizzled_scales_bytes", "nvfp4_swizzle_block_scales", "nvfp4_gemm_workspace_bytes",
    "nvfp4_gemm_nt", "nvfp4_tensor_workspace_bytes", "nvfp4_get_device_status", "nvfp4_status_string",
    "nvfp4_set_launch_config", "nvfp4_selftest_wait_timeout", "nvfp4_selftest_withhold_row",
    "nvfp4_abi_version", "library",
]

MODE_SIX = 0
MODE_FOUR_OVER_SIX = 1
MODE_FOUR_OVER_SIX_FP16 = 2
SCALE_ROW = 0
SCALE_TENSOR = 1
_MODES = {"six": MODE_SIX, "four_over_six": MODE_FOUR_OVER_SIX,
          "four_over_six_fp16": MODE_FOUR_OVER_SIX_FP16, MODE_SIX: MODE_SIX,
          MODE_FOUR_OVER_SIX: MODE_FOUR_OVER_SIX, MODE_FOUR_OVER_SIX_FP16: MODE_FOUR_OVER_SIX_FP16}
_KINDS = {"row": SCALE_ROW, "tensor": SCALE_TENSOR, SCALE_ROW: SCALE_ROW,
          SCALE_TENSOR: SCALE_TENSOR}

STATUS_NAMES = {0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_SHAPE",
                3: "NVFP4_ERR_ALIGNMENT", 4: "NVFP4_ERR_CUDA", 5: "NVFP4_ERR_TIMEOUT",
                6: "NVFP4_ERR_OFFSETS", 7: "NVFP4_ERR_WORKSPACE"}


class Nvfp4Error(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({nvfp4_status_string(status)})")


_lib = None


def library():
    """The loaded libnvfp4_gb300.so (ctypes.CDLL).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIBRARY
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (or `python -m nvfp4_block_scaled_row_gb300.build`); this package has "
            f"no fallback implementation")
    lib = ctypes.CDLL(path)
    P, I64, I32, I, SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                          ctypes.c_size_t)
    sigs = {
        "nvfp4_quantize_rowwise": [P, I64, I64, P, I32, I, P, P, P, P],
        "nvfp4_tensor_workspace_bytes": [],
        "nvfp4_quantize_tensor": [P, I64, I64, I, P, P, P, P, SZ, P],
        "nvfp4_tensor_amax": [P, I64, P, P, SZ, P],
        "nvfp4_quantize_tensor_with_amax": [P, I64, I64, I, P, P, P, P, P],
        "nvfp4_quantize_tensor_noalloc": [P, I64, I64, I, P, P, P, P],
        "nvfp4_quantize_residual": [P, I64, I64, I, P, P, P, P, P, P, P],
        "nvfp4_row_amax": [P, I64, I64, P, P],
        "nvfp4_swizzled_scales_bytes": [I64, I64],
        "nvfp4_swizzle_block_scales": [P, I64, I64, P, P],
        "nvfp4_gemm_workspace_bytes": [I64, I64],
        "nvfp4_gemm_nt": [P, P, P, P, P, P, I64, I64, I64, P, P, SZ, P],
        "nvfp4_quantize_guided": [P, I64, I64, I, P, P, P, P, P],
        "nvfp4_dequantize": [P, P, P, I, I64, I64, P, P],
        "nvfp4_fused_roundtrip": [P, I64, I64, I, I, P, P, P, P, P, SZ, P],
        "nvfp4_roundtrip_host_workspace_bytes": [I64],
        "nvfp4_fused_roundtrip_host": [P, I64, I64, I, P, P, P, P, P, SZ, P],
        "nvfp4_get_device_status": [I, P],
        "nvfp4_status_string": [I],
        "nvfp4_set_launch_config": [I, I, I],
        "nvfp4_selftest_wait_timeout": [ctypes.c_uint64, P],
        "nvfp4_selftest_withhold_row": [I64, ctypes.c_uint64],
        "nvfp4_abi_version": [],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    lib.nvfp4_tensor_workspace_bytes.restype = SZ
    lib.nvfp4_roundtrip_host_workspace_bytes.restype = SZ
    lib.nvfp4_swizzled_scales_bytes.restype = SZ
    lib.nvfp4_gemm_workspace_bytes.restype = SZ
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status, where):
    if status != 0:
        raise Nvfp4Error(status, where)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _on(device, name, *args):
    """Calls the library's `name` with `device` current: the library finds its per-device state
    (status word, multiprocessor count, the allocation-free call's array) through the current
    device, which must be the one that holds the call's tensors."""
    with torch.cuda.device(device):
        return getattr(library(), name)(*args)


def _need(t, name, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor on {device}, got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _input(x):
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a 2-D torch.Tensor [rows, cols]")
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if x.dtype != torch.bfloat16:
        raise TypeError(f"x must be torch.bfloat16, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    return x.shape[0], x.shape[1]


def _out(t, name, dtype, shape, device):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _need(t, name, dtype, shape, device)


def _workspace(workspace, device):
    n = nvfp4_tensor_workspace_bytes()
    if workspace is None:
        workspace = torch.empty(n, dtype=torch.uint8, device=device)
    elif not workspace.is_cuda or workspace.device != device:
        raise ValueError("workspace must be a CUDA tensor on the input's device")
    return workspace


def nvfp4_quantize_residual(x, mode="four_over_six", stream=None):
    """Q(x) and Q(dx), dx = bf16(x - DQ(Q(x))), both per-token 4/6, in one pass.  Returns
    ((codes, block_scales, row_scale), (res_codes, res_block_scales, res_row_scale))."""
    rows, cols = _input(x)
    dev = x.device
    outs = []
    for _ in range(2):
        outs.append((torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev),
                     torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev),
                     torch.empty((rows,), dtype=torch.float32, device=dev)))
    (c, s, d), (rc, rs, rd) = outs
    st = _on(dev, "nvfp4_quantize_residual", _ptr(x), rows, cols, _MODES[mode], _ptr(c), _ptr(s),
                                           _ptr(d), _ptr(rc), _ptr(rs), _ptr(rd),
                                           _stream(stream, dev))
    _check(st, "nvfp4_quantize_residual")
    return outs[0], outs[1]


def nvfp4_row_amax(x, row_amax=None, stream=None):
    """Per-token amax, float32 [rows]."""
    rows, cols = _input(x)
    row_amax = _out(row_amax, "row_amax", torch.float32, (rows,), x.device)
    _check(_on(x.device, "nvfp4_row_amax", _ptr(x), rows, cols, _ptr(row_amax),
               _stream(stream, x.device)), "nvfp4_row_amax")
    return row_amax


def nvfp4_quantize_guided(x, row_amax, ref_codes, ref_block_scales, mode="four_over_six",
                          codes=None, stream=None):
    """TRACE-guided codes for x under a rollout's per-token amax, codes and block scales."""
    rows, cols = _input(x)
    dev = x.device
    _need(row_amax, "row_amax", torch.float32, (rows,), dev)
    _need(ref_codes, "ref_codes", torch.uint8, (rows, cols // 2), dev)
    _need(ref_block_scales, "ref_block_scales", torch.uint8, (rows, cols // 16), dev)
    codes = _out(codes, "codes", torch.uint8, (rows, cols // 2), dev)
    st = _on(dev, "nvfp4_quantize_guided", _ptr(x), rows, cols, _MODES[mode], _ptr(row_amax),
                                         _ptr(ref_codes), _ptr(ref_block_scales), _ptr(codes),
                                         _stream(stream, dev))
    _check(st, "nvfp4_quantize_guided")
    return codes


def nvfp4_swizzled_scales_bytes(rows, cols):
    return int(library().nvfp4_swizzled_scales_bytes(int(rows), int(cols)))


def nvfp4_swizzle_block_scales(block_scales, cols, out=None, stream=None):
    """Row-major E4M3 block scales [rows, cols/16] -> the MMA-ready tiled layout (uint8, 1-D)."""
    rows = block_scales.shape[0]
    dev = block_scales.device
    _need(block_scales, "block_scales", torch.uint8, (rows, cols // 16), dev)
    n = nvfp4_swizzled_scales_bytes(rows, cols)
    out = _out(out, "out", torch.uint8, (n,), dev)
    _check(_on(dev, "nvfp4_swizzle_block_scales", _ptr(block_scales), rows, cols, _ptr(out),
                                                _stream(stream, dev)),
           "nvfp4_swizzle_block_scales")
    return out


def nvfp4_gemm_workspace_bytes(m, n):
    return int(library().nvfp4_gemm_workspace_bytes(int(m), int(n)))


def nvfp4_gemm_nt(x_codes, x_scales_swizzled, x_row_scale, w_codes, w_scales_swizzled,
                  w_tensor_scale, y=None, stream=None):
    """y[m, n] = x . w^T from NVFP4 operands (per-token x scale, per-tensor w scale), BF16."""
    m, k = x_codes.shape[0], x_codes.shape[1] * 2
    n = w_codes.shape[0]
    dev = x_codes.device
    y = _out(y, "y", torch.bfloat16, (m, n), dev)
    st = _on(dev, "nvfp4_gemm_nt", _ptr(x_codes), _ptr(x_scales_swizzled), _ptr(x_row_scale),
             _ptr(w_codes), _ptr(w_scales_swizzled), _ptr(w_tensor_scale), m, n, k, _ptr(y),
             None, 0, _stream(stream, dev))
    _check(st, "nvfp4_gemm_nt")
    return y


def nvfp4_tensor_workspace_bytes():
    return int(library().nvfp4_tensor_workspace_bytes())


def nvfp4_quantize_rowwise(x, mode="four_over_six", group_offsets=None, codes=None,
                           block_scales=None, row_scale=None, stream=None):
    """Per-token quantization.  Returns (codes [rows, cols/2] uint8, block_scales
    [rows, cols/16] uint8, row_scale [rows] float32 = S_dec)."""
    rows, cols = _input(x)
    dev = x.device
    codes = _out(codes, "codes", torch.uint8, (rows, cols // 2), dev)
    block_scales = _out(block_scales, "block_scales", torch.uint8, (rows, cols // 16), dev)
    row_scale = _out(row_scale, "row_scale", torch.float32, (rows,), dev)
    groups = 0
    if group_offsets is not None:
        if group_offsets.dim() != 1 or group_offsets.numel() < 1:
            raise ValueError("group_offsets must be 1-D with num_groups + 1 entries")
        _need(group_offsets, "group_offsets", torch.int32, group_offsets.shape, dev)
        groups = group_offsets.numel() - 1
    st = _on(dev, "nvfp4_quantize_rowwise", _ptr(x), rows, cols, _ptr(group_offsets), groups,
                                          _MODES[mode], _ptr(codes), _ptr(block_scales),
                                          _ptr(row_scale), _stream(stream, dev))
    _check(st, "nvfp4_quantize_rowwise")
    return codes, block_scales, row_scale


def nvfp4_quantize_tensor(x, mode="four_over_six", codes=None, block_scales=None,
                          tensor_scale=None, workspace=None, stream=None):
    """Per-tensor quantization.  Returns (codes, block_scales, tensor_scale [1] = S_dec)."""
    rows, cols = _input(x)
    dev = x.device
    codes = _out(codes, "codes", torch.uint8, (rows, cols // 2), dev)
    block_scales = _out(block_scales, "block_scales", torch.uint8, (rows, cols // 16), dev)
    tensor_scale = _out(tensor_scale, "tensor_scale", torch.float32, (1,), dev)
    workspace = _workspace(workspace, dev)
    st = _on(dev, "nvfp4_quantize_tensor", _ptr(x), rows, cols, _MODES[mode], _ptr(codes),
                                         _ptr(block_scales), _ptr(tensor_scale), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream, dev))
    _check(st, "nvfp4_quantize_tensor")
    return codes, block_scales, tensor_scale


def nvfp4_tensor_amax(x, amax=None, workspace=None, stream=None):
    """max |x| over a contiguous BF16 CUDA tensor, as a float32 [1] device tensor."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    dev = x.device
    amax = _out(amax, "amax", torch.float32, (1,), dev)
    workspace = _workspace(workspace, dev)
    st = _on(dev, "nvfp4_tensor_amax", _ptr(x), x.numel(), _ptr(amax), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _stream(stream, dev))
    _check(st, "nvfp4_tensor_amax")
    return amax


def nvfp4_quantize_tensor_with_amax(x, amax, mode="four_over_six", codes=None,
                                    block_scales=None, tensor_scale=None, stream=None):
    """Per-tensor quantization with a caller-supplied amax (float32 [1] device tensor)."""
    rows, cols = _input(x)
    dev = x.device
    _need(amax, "amax", torch.float32, (1,), dev)
    codes = _out(codes, "codes", torch.uint8, (rows, cols // 2), dev)
    block_scales = _out(block_scales, "block_scales", torch.uint8, (rows, cols // 16), dev)
    tensor_scale = _out(tensor_scale, "tensor_scale", torch.float32, (1,), dev)
    st = _on(dev, "nvfp4_quantize_tensor_with_amax", _ptr(x), rows, cols, _MODES[mode], _ptr(amax),
                                                   _ptr(codes), _ptr(block_scales),
                                                   _ptr(tensor_scale), _stream(stream, dev))
    _check(st, "nvfp4_quantize_tensor_with_amax")
    return codes, block_scales, tensor_scale


def nvfp4_quantize_tensor_noalloc(x, mode="four_over_six", codes=None, block_scales=None,
                                  tensor_scale=None, stream=None):
    """nvfp4_quantize_tensor without a workspace, for callers that cannot allocate: the amax
    scratch lives in a fixed device array inside the library.  Outputs that are not supplied are
    still allocated here; pass them in to keep the call allocation-free.  Calls must not overlap
    on the GPU (they share the array)."""
    rows, cols = _input(x)
    dev = x.device
    codes = _out(codes, "codes", torch.uint8, (rows, cols // 2), dev)
    block_scales = _out(block_scales, "block_scales", torch.uint8, (rows, cols // 16), dev)
    tensor_scale = _out(tensor_scale, "tensor_scale", torch.float32, (1,), dev)
    st = _on(dev, "nvfp4_quantize_tensor_noalloc", _ptr(x), rows, cols, _MODES[mode], _ptr(codes),
                                                 _ptr(block_scales), _ptr(tensor_scale),
                                                 _stream(stream, dev))
    _check(st, "nvfp4_quantize_tensor_noalloc")
    return codes, block_scales, tensor_scale


def nvfp4_dequantize(codes, block_scales, scale, kind="row", y=None, stream=None):
    """BF16 [rows, cols] = bf16(fp32(fp32(q * s) * S_dec)) from the quantizer's outputs."""
    if codes.dim() != 2:
        raise ValueError("codes must be 2-D [rows, cols/2]")
    rows, cols = codes.shape[0], codes.shape[1] * 2
    dev = codes.device
    _need(codes, "codes", torch.uint8, (rows, cols // 2), dev)
    _need(block_scales, "block_scales", torch.uint8, (rows, cols // 16), dev)
    k = _KINDS[kind]
    _need(scale, "scale", torch.float32, (rows,) if k == SCALE_ROW else (1,), dev)
    y = _out(y, "y", torch.bfloat16, (rows, cols), dev)
    st = _on(dev, "nvfp4_dequantize", _ptr(codes), _ptr(block_scales), _ptr(scale), k, rows, cols,
                                    _ptr(y), _stream(stream, dev))
    _check(st, "nvfp4_dequantize")
    return y


def nvfp4_fused_roundtrip(x, kind="row", mode="four_over_six", codes=None, block_scales=None,
                          scale=None, y=None, workspace=None, stream=None):
    """Quantize and dequantize in one pass.  Returns (codes, block_scales, scale, y)."""
    rows, cols = _input(x)
    dev = x.device
    k = _KINDS[kind]
    codes = _out(codes, "codes", torch.uint8, (rows, cols // 2), dev)
    block_scales = _out(block_scales, "block_scales", torch.uint8, (rows, cols // 16), dev)
    scale = _out(scale, "scale", torch.float32, (rows,) if k == SCALE_ROW else (1,), dev)
    y = _out(y, "y", torch.bfloat16, (rows, cols), dev)
    ws, ws_bytes = None, 0
    if k == SCALE_TENSOR:
        ws = _workspace(workspace, dev)
        ws_bytes = ws.numel() * ws.element_size()
    st = _on(dev, "nvfp4_fused_roundtrip", _ptr(x), rows, cols, k, _MODES[mode], _ptr(codes),
                                         _ptr(block_scales), _ptr(scale), _ptr(y), _ptr(ws),
                                         ws_bytes, _stream(stream, dev))
    _check(st, "nvfp4_fused_roundtrip")
    return codes, block_scales, scale, y


def nvfp4_roundtrip_host_workspace_bytes(cols):
    return int(library().nvfp4_roundtrip_host_workspace_bytes(int(cols)))


def _host(t, name, dtype, shape):
    if t.is_cuda or t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host tensor {dtype} {tuple(shape)}")
    return t


def nvfp4_fused_roundtrip_host(x, mode="four_over_six", codes=None, block_scales=None,
                               row_scale=None, y=None, workspace=None, stream=None, device=None):
    """Per-token fused round trip of a HOST bf16 matrix, streamed through the GPU.  Outputs are
    host tensors (allocated page-locked when not given).  Asynchronous on `stream`: synchronize it
    before reading the outputs."""
    if x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D bfloat16 host tensor")
    rows, cols = x.shape
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)

    def out(t, name, dtype, shape):
        if t is None:
            return torch.empty(shape, dtype=dtype, pin_memory=True)
        return _host(t, name, dtype, shape)

    codes = out(codes, "codes", torch.uint8, (rows, cols // 2))
    block_scales = out(block_scales, "block_scales", torch.uint8, (rows, cols // 16))
    row_scale = out(row_scale, "row_scale", torch.float32, (rows,))
    y = out(y, "y", torch.bfloat16, (rows, cols))
    need = nvfp4_roundtrip_host_workspace_bytes(cols)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = _on(dev, "nvfp4_fused_roundtrip_host", _ptr(x), rows, cols, _MODES[mode], _ptr(codes),
                                              _ptr(block_scales), _ptr(row_scale), _ptr(y),
                                              _ptr(workspace),
                                              workspace.numel() * workspace.element_size(),
                                              _stream(stream, dev))
    _check(st, "nvfp4_fused_roundtrip_host")
    return codes, block_scales, row_scale, y


def nvfp4_get_device_status(clear=True):
    """Synchronizes the current device; returns the device status code (0 = OK)."""
    out = ctypes.c_int(0)
    _check(library().nvfp4_get_device_status(1 if clear else 0, ctypes.byref(out)),
           "nvfp4_get_device_status")
    return out.value


def nvfp4_status_string(status):
    return library().nvfp4_status_string(int(status)).decode()


def nvfp4_set_launch_config(warps_per_cta=0, stages=0, max_ctas=0):
    _check(library().nvfp4_set_launch_config(warps_per_cta, stages, max_ctas),
           "nvfp4_set_launch_config")


def nvfp4_selftest_wait_timeout(timeout_ns=1_000_000, stream=None, device=None):
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    _check(_on(dev, "nvfp4_selftest_wait_timeout", timeout_ns, _stream(stream, dev)),
           "nvfp4_selftest_wait_timeout")


def nvfp4_selftest_withhold_row(row=-1, timeout_ns=0):
    """Test hook: quantize calls withhold row `row`'s copies and give up after timeout_ns
    (row = -1 restores normal operation)."""
    _check(library().nvfp4_selftest_withhold_row(int(row), int(timeout_ns)),
           "nvfp4_selftest_withhold_row")


def nvfp4_abi_version():
    return int(library().nvfp4_abi_version())
