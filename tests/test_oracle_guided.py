"""Pins for the oracle's TRACE-guided rounding: the page's worked example, identity when the
trainer sees the rollout's values, the choice is always a neighbouring codeword, and it never
moves further from the rollout's codeword than round-to-nearest would."""
import numpy as np
import pytest

import oracle
from conftest import read_golden
from indep import GRID, bf16_to_f64, e2m1_decode, e4m3_decode, f32_to_bf16_bits, unpack_codes
from nvfp4_block_scaled_row_gb300 import synth

F4 = oracle.MODE_FOUR_OVER_SIX
SIGNED = np.unique(np.concatenate([-GRID, GRID]))


def _rollout(xb):
    out = oracle.quantize(xb, F4)
    amax = np.array([oracle.amax(xb[r]) for r in range(xb.shape[0])], np.float32)
    return out, amax


def _trainer_view(xb, seed):
    """The training engine's slightly different activations (BF16 noise of a few ulps)."""
    rng = np.random.default_rng(seed)
    x = bf16_to_f64(xb)
    return f32_to_bf16_bits((x * (1 + rng.normal(0, 2.0 ** -7, x.shape))).astype(np.float32))


def _scaled_targets(xb, amax, scales):
    """t as the quantizer forms it (FP32: z = x * S_enc, t = z * fp32(1/s))."""
    S_enc = np.array([oracle.factors(a, F4)[0] for a in amax], np.float32)
    s = np.repeat(e4m3_decode(scales), 16, axis=1).astype(np.float32)
    inv = np.where(s > 0, np.float32(1) / np.where(s > 0, s, 1), 0).astype(np.float32)
    z = (bf16_to_f64(xb).astype(np.float32) * S_enc[:, None]).astype(np.float32)
    return (z * inv).astype(np.float32).astype(np.float64)


def test_trace_worked_example():
    (rollout, trainer, want), = [tuple(map(float, r)) for r in read_golden("trace_guided_example.txt")]

    def row(v):
        """One 16-element block with row amax 1536 (S_enc = 1) and the value in element 1."""
        r = np.zeros(16, np.float32)
        r[0], r[1] = 1536.0, v
        return f32_to_bf16_bits(r)[None, :]

    rb, tb = row(rollout), row(trainer)
    amax = np.array([1536.0], np.float32)
    scales = np.array([[0x38]], np.uint8)  # the rollout's block scale: E4M3 1.0, so t = x
    rcode = int(oracle.e2m1_encode(np.array([bf16_to_f64(rb)[0, 1]], np.float32))[0])
    ref_codes = np.zeros((1, 8), np.uint8)
    ref_codes[0, 0] = (rcode << 4) | 7  # element 0 (the 1536) maps to 6 (code 7)
    assert oracle.e2m1_value(rcode) == 3.0                       # rollout rounded to 3
    own = oracle.e2m1_encode(np.array([bf16_to_f64(tb)[0, 1]], np.float32))[0]
    assert oracle.e2m1_value(int(own)) == 2.0                    # trainer alone rounds to 2
    got = oracle.quantize_guided(tb, amax, ref_codes, scales)
    assert e2m1_decode(unpack_codes(got))[0, 1] == want          # guided by the rollout: 3


def test_identity_when_trainer_matches_rollout():
    for idx, rows in ((0, None), (2, 24), (4, 64)):
        xb = synth.as_u16(synth.generate(idx, rows=rows)["x"])
        out, amax = _rollout(xb)
        got = oracle.quantize_guided(xb, amax, out["codes"], out["scales"])
        assert np.array_equal(got, out["codes"])


@pytest.mark.parametrize("seed", [1, 2])
def test_choice_is_a_neighbour_and_never_further_than_rtn(seed):
    xb = synth.as_u16(synth.generate(2, rows=32)["x"])
    out, amax = _rollout(xb)
    xt = _trainer_view(xb, seed)
    got = oracle.quantize_guided(xt, amax, out["codes"], out["scales"])
    t = np.clip(_scaled_targets(xt, amax, out["scales"]), -6, 6)
    v = e2m1_decode(unpack_codes(got))
    ref = e2m1_decode(unpack_codes(out["codes"]))
    lo = SIGNED[np.searchsorted(SIGNED, t, side="right") - 1]
    hi = SIGNED[np.searchsorted(SIGNED, t, side="left")]
    assert np.all((v == lo) | (v == hi))
    rtn = np.where(np.abs(t - lo) < np.abs(hi - t), lo, hi)  # nearest (tie side irrelevant here)
    assert np.all(np.abs(v - ref) <= np.abs(rtn - ref))
    # and it actually changes codes where the trainer's nearest codeword disagrees
    trainer_rtn = oracle.quantize_guided(xt, amax, unpack_to_self(xt, amax, out["scales"]),
                                         out["scales"])
    assert (got != trainer_rtn).any()


def unpack_to_self(xt, amax, scales):
    """The trainer's own round-to-nearest codes under the rollout's scales (reference = itself)."""
    t = _scaled_targets(xt, amax, scales)
    codes = oracle.e2m1_encode(t.astype(np.float32))
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
