"""Python access to the C oracle (nvfp4_oracle.c) through ctypes.

TEST INFRASTRUCTURE ONLY: the plain CPU statement of the quantizer that the CUDA library is
checked against.  Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package; the library itself never does.

Inputs and outputs are numpy arrays.  BF16 tensors travel as their uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

MODE_SIX = 0
MODE_FOUR_OVER_SIX = 1
MODE_FOUR_OVER_SIX_FP16 = 2
SCALE_ROW = 0
SCALE_TENSOR = 1
BLOCK = 16

_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.oracle_e2m1_value.restype = ctypes.c_double
    lib.oracle_e2m1_value.argtypes = [I]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e4m3_value.argtypes = [I]
    lib.oracle_e2m1_encode.restype = I
    lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = I
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_bf16_encode.restype = ctypes.c_uint16
    lib.oracle_bf16_encode.argtypes = [ctypes.c_float]
    lib.oracle_factors.restype = None
    lib.oracle_factors.argtypes = [ctypes.c_float, I, P]
    lib.oracle_amax.restype = ctypes.c_float
    lib.oracle_amax.argtypes = [P, I64]
    lib.oracle_quantize.restype = I
    lib.oracle_quantize.argtypes = [P, I64, I64, I, I, P, P, P, P, P]
    lib.oracle_quantize_given_amax.restype = I
    lib.oracle_quantize_given_amax.argtypes = [P, I64, I64, I, ctypes.c_float, P, P, P]
    lib.oracle_quantize_residual.restype = I
    lib.oracle_quantize_residual.argtypes = [P, I64, I64, I, P, P, P, P, P, P]
    lib.oracle_f16_round_array.restype = None
    lib.oracle_f16_round_array.argtypes = [P, I64, P]
    lib.oracle_quantize_guided.restype = I
    lib.oracle_quantize_guided.argtypes = [P, I64, I64, I, P, P, P, P]
    lib.oracle_dequantize.restype = I
    lib.oracle_dequantize.argtypes = [P, P, P, I, I64, I64, P]
    for name in ("oracle_e2m1_encode_array", "oracle_e4m3_encode_array",
                 "oracle_bf16_encode_array"):
        getattr(lib, name).restype = None
        getattr(lib, name).argtypes = [P, I64, P]
    _lib = lib
    return lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _u16(x):
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("bf16 input must be given as uint16 bit patterns")
    return x


# ---- formats -------------------------------------------------------------------------------

def e2m1_value(code):
    return _load().oracle_e2m1_value(int(code))


def e4m3_value(byte):
    return _load().oracle_e4m3_value(int(byte))


def e2m1_encode(t):
    t = np.ascontiguousarray(t, dtype=np.float32)
    out = np.empty(t.shape, np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(t), t.size, _ptr(out))
    return out


def e4m3_encode(v):
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_encode(v):
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_bf16_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def f16_round(v):
    """The oracle's FP16 round-to-nearest-even of float64 values."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.float64)
    _load().oracle_f16_round_array(_ptr(v), v.size, _ptr(out))
    return out


# ---- the method ----------------------------------------------------------------------------

def factors(amax, mode):
    """(S_enc, c6, c4, S_dec) as float32 for one amax."""
    out = np.zeros(4, np.float32)
    _load().oracle_factors(ctypes.c_float(amax), int(mode), _ptr(out))
    return out


def amax(x_u16):
    x = _u16(x_u16)
    return float(_load().oracle_amax(_ptr(x), x.size))


def quantize(x_u16, mode=MODE_FOUR_OVER_SIX, scale_kind=SCALE_ROW, diagnostics=False):
    """Quantize a [rows, cols] BF16 matrix (uint16 bits).

    Returns a dict with ``codes`` uint8 [rows, cols/2], ``scales`` uint8 [rows, cols/16],
    ``scale`` float32 [rows] (row scale) or [1] (tensor scale) holding S_dec, and with
    ``diagnostics`` also ``choice`` uint8 [rows, cols/16] (1 = scale-to-4) and ``errs``
    float32 [rows, cols/16, 2] (e6, e4).
    """
    x = _u16(x_u16)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // BLOCK), np.uint8)
    scale = np.zeros(rows if scale_kind == SCALE_ROW else 1, np.float32)
    choice = np.zeros((rows, cols // BLOCK), np.uint8) if diagnostics else None
    errs = np.zeros((rows, cols // BLOCK, 2), np.float32) if diagnostics else None
    rc = _load().oracle_quantize(_ptr(x), rows, cols, int(mode), int(scale_kind), _ptr(codes),
                                 _ptr(scales), _ptr(scale), _ptr(choice), _ptr(errs))
    if rc:
        raise ValueError(f"oracle_quantize rejected shape {x.shape} / mode {mode}")
    out = {"codes": codes, "scales": scales, "scale": scale}
    if diagnostics:
        out["choice"] = choice
        out["errs"] = errs
    return out


def quantize_given_amax(x_u16, amax_value, mode=MODE_FOUR_OVER_SIX):
    x = _u16(x_u16)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // BLOCK), np.uint8)
    scale = np.zeros(1, np.float32)
    rc = _load().oracle_quantize_given_amax(_ptr(x), rows, cols, int(mode),
                                            ctypes.c_float(amax_value), _ptr(codes),
                                            _ptr(scales), _ptr(scale))
    if rc:
        raise ValueError("oracle_quantize_given_amax rejected its arguments")
    return {"codes": codes, "scales": scales, "scale": scale}


def quantize_residual(x_u16, mode=MODE_FOUR_OVER_SIX):
    """Q(x) and Q(dx), dx = bf16(x - DQ(Q(x))), both per-token: returns (main, residual) dicts
    shaped like quantize()'s."""
    x = _u16(x_u16)
    rows, cols = x.shape
    outs = []
    for _ in range(2):
        outs.append({"codes": np.zeros((rows, cols // 2), np.uint8),
                     "scales": np.zeros((rows, cols // BLOCK), np.uint8),
                     "scale": np.zeros(rows, np.float32)})
    a, b = outs
    rc = _load().oracle_quantize_residual(_ptr(x), rows, cols, int(mode), _ptr(a["codes"]),
                                          _ptr(a["scales"]), _ptr(a["scale"]), _ptr(b["codes"]),
                                          _ptr(b["scales"]), _ptr(b["scale"]))
    if rc:
        raise ValueError("oracle_quantize_residual rejected its arguments")
    return a, b


def quantize_guided(x_u16, row_amax, ref_codes, ref_scales, mode=MODE_FOUR_OVER_SIX):
    """TRACE-guided codes for x given the rollout's per-token amax, codes and block scales."""
    x = _u16(x_u16)
    rows, cols = x.shape
    row_amax = np.ascontiguousarray(row_amax, np.float32)
    ref_codes = np.ascontiguousarray(ref_codes, np.uint8)
    ref_scales = np.ascontiguousarray(ref_scales, np.uint8)
    out = np.zeros((rows, cols // 2), np.uint8)
    rc = _load().oracle_quantize_guided(_ptr(x), rows, cols, int(mode), _ptr(row_amax),
                                        _ptr(ref_codes), _ptr(ref_scales), _ptr(out))
    if rc:
        raise ValueError("oracle_quantize_guided rejected its arguments")
    return out


def dequantize(codes, scales, scale, scale_kind=SCALE_ROW):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    scale = np.ascontiguousarray(scale, np.float32)
    rows, half = codes.shape
    cols = half * 2
    y = np.zeros((rows, cols), np.uint16)
    rc = _load().oracle_dequantize(_ptr(codes), _ptr(scales), _ptr(scale), int(scale_kind),
                                   rows, cols, _ptr(y))
    if rc:
        raise ValueError("oracle_dequantize rejected its arguments")
    return y


def library_path():
    return os.path.abspath(_build.LIBRARY)
