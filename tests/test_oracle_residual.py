"""Pins for the oracle's residual quantization (Rollout-ResQ with NVFP4 per-token 4/6): it is the
composition of the separately pinned quantizer and dequantizer with an independently computed
BF16 residual, it vanishes on grid values, and it recovers most of what the main term loses."""
import numpy as np
import pytest

import oracle
from indep import bf16_to_f64, exact_dequant, f32_to_bf16_bits
from nvfp4_block_scaled_row_gb300 import synth

F4, SIX = oracle.MODE_FOUR_OVER_SIX, oracle.MODE_SIX


@pytest.fixture(scope="module")
def inputs():
    return [synth.as_u16(synth.generate(0)["x"]), synth.as_u16(synth.generate(2, rows=40)["x"]),
            synth.as_u16(synth.generate(4, rows=120)["x"])]


@pytest.mark.parametrize("mode", [F4, SIX])
def test_residual_is_quantize_of_independent_residual(inputs, mode):
    for xb in inputs:
        main, res = oracle.quantize_residual(xb, mode)
        want = oracle.quantize(xb, mode)
        for k in ("codes", "scales", "scale"):
            assert np.array_equal(main[k], want[k])
        y = bf16_to_f64(oracle.dequantize(want["codes"], want["scales"], want["scale"]))
        x = bf16_to_f64(xb)
        dx = f32_to_bf16_bits((x.astype(np.float32) - y.astype(np.float32)).astype(np.float32))
        want_r = oracle.quantize(dx, mode)
        for k in ("codes", "scales", "scale"):
            assert np.array_equal(res[k], want_r[k])


def test_residual_vanishes_on_grid_values():
    # Rows whose values are exactly representable by the main term leave a zero residual.
    rng = np.random.default_rng(3)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    rows = []
    for k in (-4, 0, 7):
        q = grid[rng.integers(0, 8, 256)] * np.where(rng.integers(0, 2, 256), -1, 1)
        q[::16] = 6.0  # every block's max maps exactly to 6
        rows.append(q * 2.0 ** k)
    xb = f32_to_bf16_bits(np.array(rows, np.float32))
    main, res = oracle.quantize_residual(xb)
    assert np.array_equal(oracle.dequantize(main["codes"], main["scales"], main["scale"]), xb)
    assert not res["codes"].any() and not res["scales"].any() and not res["scale"].any()


def test_residual_recovers_most_of_the_error(inputs):
    for xb in inputs:
        main, res = oracle.quantize_residual(xb)
        x = bf16_to_f64(xb)
        y1 = exact_dequant(main, xb.shape[1])
        y2 = exact_dequant(res, xb.shape[1])
        e1 = np.sqrt(np.mean((x - y1) ** 2))
        e2 = np.sqrt(np.mean((x - y1 - y2) ** 2))
        assert e2 <= 0.25 * e1
        lost = (y1 == 0) & (x != 0)  # small values the main term flushed to zero
        if lost.sum() > 100:
            assert np.mean(y2[lost] != 0) > 0.5
