"""Independent checks used by the oracle pins.

Nothing here calls the oracle's arithmetic: decoding goes through the page's E2M1 grid and
torch's float8_e4m3fn / bfloat16 conversions (library routines), and exact values are formed in
float64, where every product below is exact.
"""
import numpy as np
import torch

from conftest import read_golden

GRID = np.array([float(r[0]) for r in read_golden("e2m1_grid.txt")], np.float64)


def e2m1_decode(codes_nibbles):
    c = np.asarray(codes_nibbles, np.int64)
    mag = GRID[c & 7]
    return np.where(c & 8, -mag, mag)


def unpack_codes(packed):
    """[rows, cols/2] bytes -> [rows, cols] nibbles, element 2j in the low nibble of byte j."""
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def e4m3_decode(bytes_):
    b = torch.from_numpy(np.ascontiguousarray(bytes_, np.uint8))
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e4m3_round(values_f32):
    """torch's float32 -> float8_e4m3fn (round to nearest even) as bytes; valid up to 464."""
    v = torch.from_numpy(np.ascontiguousarray(values_f32, np.float32))
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def bf16_to_f64(u16):
    u = np.asarray(u16, np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(v_f32):
    v = torch.from_numpy(np.ascontiguousarray(v_f32, np.float32))
    return v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def exact_dequant(out, cols):
    """float64 value of every encoded element: r * s * S_dec (row scale), exact in float64."""
    r = e2m1_decode(unpack_codes(out["codes"]))
    s = np.repeat(e4m3_decode(out["scales"]), 16, axis=-1)
    scale = out["scale"].astype(np.float64)
    sd = scale[:, None] if scale.shape[0] == r.shape[0] else scale[0]
    return r * s * sd
