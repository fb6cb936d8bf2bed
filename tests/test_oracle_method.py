"""Pins for the oracle's quantizer: what the pages and plain mathematics fix about its output.

Each check recomputes what it needs independently (tests/indep.py: the page's E2M1 grid, torch's
FP8/BF16 conversions, float64), so a dropped term, a wrong sign or index, or a swapped operand in
the oracle fails one of them.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from indep import (GRID, bf16_to_f64, e2m1_decode, e4m3_decode, e4m3_round, exact_dequant,
                   f32_to_bf16_bits, unpack_codes)
from nvfp4_block_scaled_row_gb300 import synth

F4 = oracle.MODE_FOUR_OVER_SIX
SIX = oracle.MODE_SIX


def _bits(a_f32):
    return f32_to_bf16_bits(np.asarray(a_f32, np.float32))


def _inputs():
    """Workload 0 at full size and small instances of workloads 1-4 (same recipes)."""
    cases = [synth.generate(0)["x"], synth.generate(1, rows=48)["x"], synth.generate(2, rows=48)["x"],
             synth.generate(3, rows=640)["x"], synth.generate(4, rows=200)["x"]]
    return [synth.as_u16(x) for x in cases]


@pytest.fixture(scope="module")
def inputs():
    return _inputs()


def _bound_fraction():
    return {int(r[0]): eval(r[1], {}) for r in read_golden("four_over_six_bounds.txt")}


@pytest.mark.parametrize("mode", [F4, SIX])
def test_worst_case_error_bounds(inputs, mode):
    """Every block: |x - DQ(Q(x))| <= range/6 when mapped to 6 and <= range/8 when mapped to 4,
    where range = T * s * S_dec is the value the block max is mapped to."""
    frac = _bound_fraction()
    for kind in (oracle.SCALE_ROW, oracle.SCALE_TENSOR):
        for xb in inputs:
            out = oracle.quantize(xb, mode, kind, diagnostics=True)
            rows, cols = xb.shape
            x = bf16_to_f64(xb).reshape(rows, cols // 16, 16)
            y = exact_dequant(out, cols).reshape(rows, cols // 16, 16)
            T = np.where(out["choice"] == 1, 4, 6)
            s = e4m3_decode(out["scales"])
            sd = out["scale"].astype(np.float64)
            sd = sd[:, None] if kind == oracle.SCALE_ROW else sd[0]
            rng = T * s * sd
            bound = np.where(T == 4, frac[4], frac[6]) * rng
            err = np.abs(x - y).max(axis=2)
            live = s > 0
            assert np.all(err[live] <= bound[live] * (1 + 2.0 ** -20) + 1e-45)
            # A zero block scale encodes all zeros; that only happens when the block's scale
            # underflowed E4M3, i.e. when m * c_T < 2^-10.
            assert np.all(y[~live] == 0)


def test_page_example_five_sixths_prefers_four():
    """The pages' motivating case: values near 5/6 of the range are off by 1/6 of the range when
    the max maps to 6, and 4/6 then maps the max to 4 instead."""
    a = np.float32(1536.0)  # S_enc = 1 for mode four_over_six
    row = np.full(16, 1280.0, np.float32)  # 5/6 of the block max
    row[0] = 1536.0
    xb = _bits(np.tile(row, 4))[None, :]
    six = oracle.quantize(xb, SIX, diagnostics=True)
    x = bf16_to_f64(xb)
    y6 = exact_dequant(six, 64)
    rng6 = 6 * e4m3_decode(six["scales"])[0, 0] * six["scale"][0]
    assert np.isclose(np.abs(x - y6).max(), rng6 / 6, rtol=1e-6)
    f46 = oracle.quantize(xb, F4, diagnostics=True)
    assert np.all(f46["choice"] == 1)
    y4 = exact_dequant(f46, 64)
    rng4 = 4 * e4m3_decode(f46["scales"])[0, 0] * f46["scale"][0]
    assert np.abs(x - y4).max() <= rng4 / 8
    assert a == np.float32(np.abs(x).max())


def _fp64_block_errors(xb, mode):
    """Both candidates' block squared errors recomputed in float64 in the x domain.

    The two candidate block scales are formed as the spec forms them (FP32 products m * c_T,
    rounded by torch's E4M3 conversion), so the candidates match the oracle's; the targets, the
    nearest codewords and the squared errors are then taken in float64 and compared there."""
    rows, cols = xb.shape
    M = np.float32(256.0 if mode == F4 else 448.0)
    x = bf16_to_f64(xb).reshape(rows, cols // 16, 16)
    a = np.abs(x).reshape(rows, -1).max(axis=1).astype(np.float32)
    safe = np.where(a > 0, a, np.float32(1.0)).astype(np.float32)
    m = np.abs(x).max(axis=2).astype(np.float32)
    errs = {}
    for T, c in ((6, M / safe), (4, np.float32(1.5) * M / safe)):
        u = (m * c.astype(np.float32)[:, None]).astype(np.float32)
        s = e4m3_decode(e4m3_round(u))
        sd = safe.astype(np.float64) / (6 * float(M))
        t = np.where(s[..., None] > 0, x / sd[:, None, None] / np.where(s > 0, s, 1)[..., None], 0)
        mag = np.minimum(np.abs(t), 6.0)
        idx = np.abs(mag[..., None] - GRID).argmin(axis=-1)
        r = np.sign(t) * GRID[idx]
        y = r * s[..., None] * sd[:, None, None]
        errs[T] = ((x - y) ** 2).sum(axis=2)
    return errs[6], errs[4]


def test_four_over_six_choice_agrees_with_float64(inputs):
    """The FP32 choice picks the candidate with the lower float64 block error, except in near ties
    (relative gap below 1e-3), and agrees on far more than 99.97% of blocks."""
    agree = total = 0
    for xb in inputs:
        out = oracle.quantize(xb, F4, diagnostics=True)
        e6, e4 = _fp64_block_errors(xb, F4)
        want = e4 < e6
        got = out["choice"] == 1
        gap = np.abs(e4 - e6) / np.maximum(np.maximum(e4, e6), 1e-300)
        bad = (want != got) & (gap > 1e-3)
        assert not bad.any(), f"{bad.sum()} blocks chose the worse candidate"
        agree += int((want == got).sum())
        total += want.size
    assert agree / total > 0.9997


def test_chosen_candidate_error_is_reported_minimum(inputs):
    for xb in inputs[:2]:
        out = oracle.quantize(xb, F4, diagnostics=True)
        e6, e4 = out["errs"][..., 0], out["errs"][..., 1]
        assert np.array_equal(out["choice"] == 1, e4 < e6)


def test_ties_go_to_six():
    # All-zero block: both errors 0.  Block of +-max: both candidates exact.  Both pick 6.
    zero = np.zeros(16, np.float32)
    pm = np.array([1536.0, -1536.0] * 8, np.float32)
    grid6 = np.array([1536.0, 768.0, 384.0, 0.0] * 4, np.float32)  # 6, 3, 1.5, 0 on both grids
    xb = _bits(np.concatenate([zero, pm, grid6]))[None, :]
    out = oracle.quantize(xb, F4, diagnostics=True)
    assert list(out["choice"][0]) == [0, 0, 0]
    assert np.all(out["errs"][0, 1:] == 0)
    assert out["scales"][0, 0] == 0


def chain_order_row():
    """One row of two blocks whose 4/6 choice is decided by the order of the error sum.

    The row amax is 1536, so in mode four_over_six S_enc = 6 * 256 / 1536 = 1 and the targets are
    the inputs themselves.  Both blocks hold the max (block scales: scale-to-6 256, scale-to-4 384,
    so the candidate grids are {0, 128, 256, 384, 512, 768, 1024, 1536} and {0, 192, 384, 576,
    768, 1152, 1536}), thirteen values eps = 2^-7 (zero codes under both candidates, residual eps),
    and the pair 576, 512: 576 is on the scale-to-4 grid and 64 from the scale-to-6 grid, 512 the
    other way round.  Block 0 is [576, 1536, eps x 13, 512], block 1 the mirror [512, 1536, eps x
    13, 576].  So each block has one residual of 64 and thirteen of eps under each candidate: the
    exact sums are equal (4096 + 13 * 2^-14), and only the FP32 rounding of the chain separates
    them.  The FP32 ulp at 4096 is 2^-11 = 8 * 2^-14:
      - a chain that meets the 64 first stays at 4096 (each eps^2 = 2^-14 is an eighth of an ulp);
      - a chain that meets it last adds 4096 to 13 * 2^-14 = 1.625 ulp once, giving 4096 + 2^-10.
    Summed in ascending element order, block 0's scale-to-6 chain meets its 64 first and its
    scale-to-4 chain meets it last, so e6 = 4096 < e4 = 4096 + 2^-10 and 6 is chosen; block 1 is
    the other way round and chooses 4.  Descending order reverses both choices; four interleaved
    chains over every second element of each half (combined pairwise) tie block 1 and send it to 6.
    """
    eps = 2.0 ** -7
    b0 = [576.0, 1536.0] + [eps] * 13 + [512.0]
    b1 = [512.0, 1536.0] + [eps] * 13 + [576.0]
    return _bits(np.array(b0 + b1, np.float32))[None, :]


def test_block_error_is_one_ascending_chain():
    """The block error is e = fma(d_i, d_i, e) over i = 0..15 from +0: the closed-form values of
    chain_order_row (derived in its docstring) pin the order, the choices and the error bits."""
    xb = chain_order_row()
    out = oracle.quantize(xb, F4, diagnostics=True)
    assert out["scale"][0] == np.float32(1536.0 / 1536.0)
    assert list(out["choice"][0]) == [0, 1]
    lo, hi = np.float32(4096.0), np.float32(4096.0 + 2.0 ** -10)
    assert out["errs"][0, 0].tolist() == [lo, hi]
    assert out["errs"][0, 1].tolist() == [hi, lo]
    # Scale bytes: E4M3 256 = 0x78 (scale-to-6) for block 0, E4M3 384 = 0x7C (scale-to-4) for 1.
    assert list(out["scales"][0]) == [0x78, 0x7C]
    nib = unpack_codes(out["codes"])[0]
    assert list(nib[:16]) == [4, 7] + [0] * 13 + [4]    # 576 -> 2 * 256, 1536 -> 6, 512 -> 2
    assert list(nib[16:]) == [3, 6] + [0] * 13 + [3]    # 512, 576 -> 1.5 * 384, 1536 -> 4 * 384


def test_per_element_codes_are_nearest(inputs):
    """Given the chosen scale, every code is the nearest codeword to the scaled target."""
    xb = inputs[0][:64]
    out = oracle.quantize(xb, F4, diagnostics=True)
    rows, cols = xb.shape
    S_enc = np.array([oracle.factors(oracle.amax(xb[r]), F4)[0] for r in range(rows)], np.float32)
    s = np.repeat(e4m3_decode(out["scales"]), 16, axis=1).astype(np.float32)
    x = bf16_to_f64(xb).astype(np.float32)
    z = (x * S_enc[:, None]).astype(np.float32)
    inv = np.where(s > 0, (np.float32(1) / np.where(s > 0, s, 1)).astype(np.float32), 0).astype(np.float32)
    t = (z * inv).astype(np.float64)
    r = e2m1_decode(unpack_codes(out["codes"]))
    dist = np.abs(np.minimum(np.abs(t), 6.0) - np.abs(r))
    best = np.abs(np.minimum(np.abs(t), 6.0)[..., None] - GRID).min(axis=-1)
    assert np.all(dist == best)
    assert np.all((r == 0) | (np.sign(r) == np.sign(t)))


def test_batch_independence(inputs):
    """Per-token scales keep a token's quantization independent of the rest of the batch."""
    xb = inputs[2]
    base = oracle.quantize(xb, F4)
    rng = np.random.default_rng(5)
    perm = rng.permutation(xb.shape[0])
    extra = np.ascontiguousarray(xb[:5, ::-1])  # other tokens: the first rows, reversed
    variants = {
        "permuted": (xb[perm], perm),
        "appended": (np.concatenate([xb, extra]), np.arange(xb.shape[0])),
        "dropped": (xb[::3], np.arange(0, xb.shape[0], 3)),
    }
    for name, (xv, idx) in variants.items():
        out = oracle.quantize(np.ascontiguousarray(xv), F4)
        n = len(idx)
        for key in ("codes", "scales", "scale"):
            assert np.array_equal(out[key][:n], base[key][idx]), name


def test_tensor_scale_equals_row_scale_on_one_row(inputs):
    xb = inputs[0][3:4]
    row = oracle.quantize(xb, F4, oracle.SCALE_ROW)
    ten = oracle.quantize(xb, F4, oracle.SCALE_TENSOR)
    for key in ("codes", "scales", "scale"):
        assert np.array_equal(row[key], ten[key])


def _grid_row(rng, k, four):
    """A row whose every value lies on its block's grid, with row amax 6 * 2^k.

    Scale-to-6 blocks hold q * 2^(k+j) with q on the E2M1 grid and max 6 * 2^(k+j); scale-to-4
    blocks hold q * 1.5 * 2^(k+j) with q on the grid up to 4, max 4 * 1.5 * 2^(k+j), and at least
    one value that the scale-to-6 grid cannot represent."""
    blocks, codes, picks = [], [], []
    for b in range(8):
        j = -int(rng.integers(0, 6)) if b else 0
        use4 = four and b % 2 == 1
        top = 6 if use4 else 7          # largest code index allowed
        q = rng.integers(0, top + 1, 16)
        q[rng.integers(0, 16)] = top
        if use4:
            q[(np.nonzero(q != top)[0][:1])] = 1   # 0.5 * 1.5 = 0.75: off the scale-to-6 grid
        sign = rng.integers(0, 2, 16) * 8
        sign[q == 0] = 0
        mult = 1.5 if use4 else 1.0
        vals = np.where(sign == 8, -1, 1) * GRID[q] * mult * 2.0 ** (k + j)
        blocks.append(vals)
        codes.append(q | sign)
        picks.append(int(use4))
    return np.concatenate(blocks).astype(np.float32), np.concatenate(codes), picks


@pytest.mark.parametrize("four", [False, True])
def test_idempotent_on_grid_values(four):
    """Quantize-then-dequantize returns values that are already on the grid unchanged, with the
    codes and the scale-to-4 / scale-to-6 choice known in closed form."""
    rng = np.random.default_rng(17 + four)
    rows = [_grid_row(rng, k, four) for k in (-12, -3, 0, 4, 9)]
    x = np.stack([r[0] for r in rows])
    xb = _bits(x)
    assert np.array_equal(bf16_to_f64(xb), x.astype(np.float64))
    out = oracle.quantize(xb, F4, diagnostics=True)
    y = oracle.dequantize(out["codes"], out["scales"], out["scale"])
    assert np.array_equal(y, xb)
    assert np.array_equal(unpack_codes(out["codes"]), np.stack([r[1] for r in rows]).astype(np.uint8))
    assert np.array_equal(out["choice"], np.array([r[2] for r in rows], np.uint8))
    for i, k in enumerate((-12, -3, 0, 4, 9)):
        assert out["scale"][i] == np.float32(6 * 2.0 ** k / 1536)  # S_dec = a / (6M), exact


def test_mode_six_maps_row_max_to_six(inputs):
    xb = inputs[0]
    out = oracle.quantize(xb, SIX)
    r = e2m1_decode(unpack_codes(out["codes"]))
    x = bf16_to_f64(xb)
    arg = np.abs(x).argmax(axis=1)
    rows = np.arange(x.shape[0])
    assert np.all(np.abs(r[rows, arg]) == 6.0)
    assert np.all(e4m3_decode(out["scales"])[rows, arg // 16] == 448.0)


def test_zero_rows():
    xb = np.zeros((3, 64), np.uint16)
    xb[1] = _bits(np.linspace(-3, 3, 64))
    out = oracle.quantize(xb, F4)
    for r in (0, 2):
        assert not out["codes"][r].any() and not out["scales"][r].any() and out["scale"][r] == 0
    y = oracle.dequantize(out["codes"], out["scales"], out["scale"])
    assert not y[0].any() and not y[2].any()


def test_dequant_closed_form(inputs):
    """y = bf16(fp32(fp32(q * s) * S_dec)), built from the page grid, torch's E4M3 decode, numpy
    float32 products and torch's BF16 rounding."""
    for kind in (oracle.SCALE_ROW, oracle.SCALE_TENSOR):
        for xb in inputs[:3]:
            out = oracle.quantize(xb, F4, kind)
            y = oracle.dequantize(out["codes"], out["scales"], out["scale"], kind)
            q = e2m1_decode(unpack_codes(out["codes"])).astype(np.float32)
            s = np.repeat(e4m3_decode(out["scales"]), 16, axis=1).astype(np.float32)
            sd = out["scale"][:, None] if kind == oracle.SCALE_ROW else out["scale"][0]
            want = f32_to_bf16_bits((q * s).astype(np.float32) * np.float32(sd))
            assert np.array_equal(y, want)


def test_dequant_within_half_ulp_of_exact_value(inputs):
    """DQ(Q(x)) is the exact encoded value up to one FP32 and one BF16 rounding."""
    xb = inputs[4]
    out = oracle.quantize(xb, F4)
    y = bf16_to_f64(oracle.dequantize(out["codes"], out["scales"], out["scale"]))
    exact = exact_dequant(out, xb.shape[1])
    tol = np.abs(exact) * (2.0 ** -8 + 2.0 ** -23) + 1e-44
    assert np.all(np.abs(y - exact) <= tol)


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((2, 24), np.uint16))
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((2, 32), np.uint16), mode=7)
