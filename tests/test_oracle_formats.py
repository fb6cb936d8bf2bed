"""Pins for the oracle's number formats (E2M1, E4M3, BF16) against the pages and library routines."""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from indep import GRID


def test_e2m1_decode_matches_page_grid(e2m1_grid):
    # Codes 0..7 are the page's magnitudes in order; codes 8..15 are their negatives.
    assert [oracle.e2m1_value(c) for c in range(8)] == e2m1_grid
    for c in range(8):
        v = oracle.e2m1_value(c + 8)
        assert v == -e2m1_grid[c] and np.signbit(v)


def test_e2m1_step_of_two_between_four_and_six(e2m1_grid):
    # "step size 2 between 4 and 6": the top two codewords.
    assert e2m1_grid[-1] - e2m1_grid[-2] == 2


def test_trace_worked_example():
    rows = read_golden("trace_worked_example.txt")
    t = np.array([float(r[0]) for r in rows], np.float32)
    want = [float(r[1]) for r in rows]
    got = [oracle.e2m1_value(c) for c in oracle.e2m1_encode(t)]
    assert got == want


def _brute_force_e2m1(t):
    """Nearest of the eight page magnitudes, ties to the even code, sign of t kept; magnitudes
    beyond the largest codeword saturate to it."""
    t = np.asarray(t, np.float32)
    mag = np.minimum(np.abs(t.astype(np.float64)), GRID[-1])
    err = np.abs(mag[:, None] - GRID[None, :])
    best = err.min(axis=1, keepdims=True)
    cand = err == best
    # among tied codes prefer the even one (codes are 0..7, ties only between neighbours)
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    return (pick | np.where(np.signbit(t), 8, 0)).astype(np.uint8)


def _e2m1_probe_values():
    mids = (GRID[1:] + GRID[:-1]) / 2
    pts = np.concatenate([GRID, mids, [7.0, 8.0, 100.0, 1e30, 6.5, 0.0]]).astype(np.float32)
    near = np.concatenate([np.nextafter(pts, np.float32(np.inf)), np.nextafter(pts, np.float32(0))])
    rng = np.random.default_rng(7)
    rand = np.concatenate([rng.uniform(0, 8, 200000), rng.uniform(0, 1e-3, 1000),
                           np.exp(rng.uniform(-40, 40, 5000))]).astype(np.float32)
    v = np.concatenate([pts, near, rand])
    return np.concatenate([v, -v]).astype(np.float32)


def test_e2m1_encode_brute_force():
    t = _e2m1_probe_values()
    np.testing.assert_array_equal(oracle.e2m1_encode(t), _brute_force_e2m1(t))


def test_e2m1_ties_go_to_even_mantissa():
    # Halfway points between neighbouring codewords and the codeword each one rounds to.
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    t = np.array(list(ties), np.float32)
    got = [oracle.e2m1_value(c) for c in oracle.e2m1_encode(t)]
    assert got == list(ties.values())


def test_e2m1_saturates_and_keeps_sign():
    codes = oracle.e2m1_encode(np.array([6.9, 7.0, 1e9, -1e9, -0.1, -0.0, 0.0], np.float32))
    assert list(codes) == [7, 7, 7, 15, 8, 8, 0]


def test_e4m3_decode_matches_torch():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_value(i) for i in range(256)])
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert set(np.nonzero(np.isnan(ours))[0]) == {0x7F, 0xFF}
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(1) == 2.0 ** -9


def _e4m3_probe_values():
    vals = np.array([oracle.e4m3_value(b) for b in range(127)], np.float64)
    mids = (vals[1:] + vals[:-1]) / 2
    pts = np.concatenate([vals, mids, [2.0 ** -10, 3 * 2.0 ** -11, 464.0]]).astype(np.float32)
    near = np.concatenate([np.nextafter(pts, np.float32(np.inf)), np.nextafter(pts, np.float32(0))])
    rng = np.random.default_rng(11)
    rand = np.concatenate([rng.uniform(0, 464, 200000),
                           np.exp(rng.uniform(np.log(1e-6), np.log(464), 200000))]).astype(np.float32)
    v = np.concatenate([pts, near, rand])
    return v[(v >= 0) & (v <= 464)].astype(np.float32)


def test_e4m3_encode_matches_torch_in_range():
    v = _e4m3_probe_values()
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


def test_e4m3_encode_saturates_above_range():
    v = np.array([464.5, 480.0, 1e6, 3.4e38], np.float32)
    assert list(oracle.e4m3_encode(v)) == [0x7E] * 4


def test_bf16_encode_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    specials = np.array([0.0, -0.0, 1e-45, -1e-45, 1.1754942e-38, 3.4028235e38, -3.4028235e38,
                         3.3961776e38, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], np.float32)
    v = np.concatenate([v, specials]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_encode(v), ref)


@pytest.mark.parametrize("mode,M", [(oracle.MODE_FOUR_OVER_SIX, 256.0), (oracle.MODE_SIX, 448.0)])
def test_factors_power_of_two_amax_are_exact(mode, M):
    # With a = 6M * 2^k the encode scale is exactly 2^-k and the stored decode scale exactly 2^k.
    for k in (-20, -3, 0, 5, 30):
        a = np.float32(6 * M * 2.0 ** k)
        S_enc, c6, c4, S_dec = oracle.factors(a, mode)
        assert S_enc == np.float32(2.0 ** -k) and S_dec == np.float32(2.0 ** k)
        assert abs(float(c6) * 6 * 2.0 ** k - 1) < 2 ** -23
        if mode == oracle.MODE_FOUR_OVER_SIX:
            assert c4 == np.float32(2.0 ** -k / 4)


def test_factors_zero_and_tiny_amax():
    assert list(oracle.factors(0.0, oracle.MODE_FOUR_OVER_SIX)) == [0, 0, 0, 0]
    # a = 2^-118: 1536/a overflows FP32 and is clamped; 256/a and 384/a stay finite; a/1536 is
    # an FP32 subnormal but not zero.
    S_enc, c6, c4, S_dec = oracle.factors(np.float32(2.0 ** -118), oracle.MODE_FOUR_OVER_SIX)
    assert S_enc == np.finfo(np.float32).max
    assert c6 == np.float32(2.0 ** 126) and c4 == np.float32(1.5 * 2.0 ** 126)
    assert 0 < S_dec < np.finfo(np.float32).tiny
    S_enc, c6, c4, _ = oracle.factors(np.float32(2.0 ** -126), oracle.MODE_FOUR_OVER_SIX)
    assert S_enc == c6 == c4 == np.finfo(np.float32).max


def _f32_nearest(q):
    """Correctly rounded float32 of an exact rational (ties to even), by comparing the two float32
    neighbours of the float64 approximation in exact arithmetic."""
    from fractions import Fraction

    x = np.float32(float(q))
    lo, hi = (x, np.nextafter(x, np.float32(np.inf))) if Fraction(float(x)) <= q else \
             (np.nextafter(x, np.float32(-np.inf)), x)
    dl, dh = q - Fraction(float(lo)), Fraction(float(hi)) - q
    if dl < dh:
        return lo
    if dh < dl:
        return hi
    return lo if (lo.view(np.uint32) & 1) == 0 else hi


@pytest.mark.parametrize("mode,M", [(oracle.MODE_FOUR_OVER_SIX, 256), (oracle.MODE_SIX, 448)])
def test_factors_are_correctly_rounded_quotients(mode, M):
    """S_enc = 6M/a, c6 = M/a, c4 = 1.5M/a and S_dec = a/(6M), each the correctly rounded FP32
    value of the exact quotient (the candidate formula's amax / (E2M1_MAXVAL * M))."""
    from fractions import Fraction

    rng = np.random.default_rng(21)
    amaxes = (rng.standard_normal(400) * np.exp(rng.uniform(-30, 30, 400))).astype(np.float32)
    for a in np.abs(amaxes[amaxes != 0]):
        fa = Fraction(float(a))
        S_enc, c6, c4, S_dec = oracle.factors(a, mode)
        assert S_enc == _f32_nearest(Fraction(6 * M) / fa)
        assert c6 == _f32_nearest(Fraction(M) / fa)
        assert c4 == _f32_nearest(Fraction(3 * M, 2) / fa)
        assert S_dec == _f32_nearest(fa / (6 * M))
