"""Full-size GPU parity: every element of the three large workloads against the oracle.

The oracle runs on all host cores (contiguous row ranges on threads; its ctypes calls release the
GIL).  Every row of moe_activation (16384x7168), expert_grouped (~32853x7168, with its group
offsets) and long_rollout (131072x7168) is compared bit for bit -- codes, E4M3 block scales, FP32
row scales and dequantized BF16 -- with the library in its default launch configuration (the one
the benchmark times).  moe_activation is also checked in mode six, with the FP16 selector, for the
ResQ residual and for TRACE guidance, and the fused round trip's work-unit hand-over on a
3653-row instance under several grid caps.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import nvfp4_block_scaled_row_gb300 as nv
from nvfp4_block_scaled_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
OMODE = {"four_over_six": oracle.MODE_FOUR_OVER_SIX, "six": oracle.MODE_SIX,
         "four_over_six_fp16": oracle.MODE_FOUR_OVER_SIX_FP16}


@pytest.fixture(scope="module", autouse=True)
def _library():
    nv.library()
    nv.nvfp4_set_launch_config(0, 0, 0)
    nv.nvfp4_get_device_status(clear=True)
    yield
    torch.cuda.empty_cache()


def _threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def _row_ranges(rows):
    n = min(_threads(), max(1, rows))
    bounds = [rows * i // n for i in range(n + 1)]
    return [(bounds[i], bounds[i + 1]) for i in range(n) if bounds[i + 1] > bounds[i]]


def _parallel(fn, rows):
    with ThreadPoolExecutor(len(_row_ranges(rows))) as ex:
        list(ex.map(fn, _row_ranges(rows)))


def oracle_quantize_rows(xb, mode, want_y=False):
    """The oracle's per-token quantization (and dequantization) of every row of xb."""
    rows, cols = xb.shape
    out = {"codes": np.empty((rows, cols // 2), np.uint8),
           "scales": np.empty((rows, cols // 16), np.uint8),
           "scale": np.empty(rows, np.float32)}
    if want_y:
        out["y"] = np.empty((rows, cols), np.uint16)

    def one(r):
        a, b = r
        q = oracle.quantize(xb[a:b], OMODE[mode], oracle.SCALE_ROW)
        for k in ("codes", "scales", "scale"):
            out[k][a:b] = q[k]
        if want_y:
            out["y"][a:b] = oracle.dequantize(q["codes"], q["scales"], q["scale"])

    _parallel(one, rows)
    return out


def assert_same(got, want, what):
    """Exact equality of two large arrays (FP32 compared by bit pattern), checked in row slices."""
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    if got.dtype == np.float32:
        got, want = got.view(np.uint32), want.view(np.uint32)
    step = max(1, (1 << 26) // max(1, got[0].size if got.ndim > 1 else 1))
    for a in range(0, got.shape[0], step):
        g, w = got[a:a + step], want[a:a + step]
        if not np.array_equal(g, w):
            bad = np.argwhere(g != w)
            i = tuple(bad[0])
            first = (a + i[0],) + i[1:]
            raise AssertionError(f"{what}: {len(bad)} mismatches in rows {a}..{a + len(g) - 1}, "
                                 f"first at {first}: gpu={g[i]!r} oracle={w[i]!r}")


def _np(t):
    return t.detach().cpu().numpy()


def _u16(t):
    return synth.as_u16(t)


def test_moe_activation_fused_roundtrip_every_row():
    x = synth.generate(2, device=DEV)["x"]
    want = oracle_quantize_rows(_u16(x), "four_over_six", want_y=True)
    codes, scales, sdec, y = nv.nvfp4_fused_roundtrip(x, "row", "four_over_six")
    assert_same(_np(codes), want["codes"], "codes")
    assert_same(_np(scales), want["scales"], "block scales")
    assert_same(_np(sdec), want["scale"], "row scale")
    assert_same(_u16(y), want["y"], "y")
    assert nv.nvfp4_get_device_status() == 0


def test_fused_work_units_taken_over_every_row():
    """The fused round trip's dynamic schedule: one CTA per work unit (a row for each team of a
    CTA), and running CTAs take over the units of CTAs that have not started; under a grid cap each
    CTA walks every cap-th unit and takes over whole walks.  3653 rows: the units outnumber one
    wave of resident CTAs three times over and the last unit is partial; caps just above one wave,
    between one and two, and at two waves.  Every row, every cap, against the same oracle result."""
    rows = 8 * 152 * 3 + 5
    x = synth.generate(2, device=DEV, rows=rows)["x"]
    want = oracle_quantize_rows(_u16(x), "four_over_six", want_y=True)
    try:
        for cap in (0, 153, 200, 304):
            nv.nvfp4_set_launch_config(0, 0, cap)
            codes, scales, sdec, y = nv.nvfp4_fused_roundtrip(x, "row", "four_over_six")
            assert_same(_np(codes), want["codes"], f"codes (cap {cap})")
            assert_same(_np(scales), want["scales"], f"block scales (cap {cap})")
            assert_same(_np(sdec), want["scale"], f"row scale (cap {cap})")
            assert_same(_u16(y), want["y"], f"y (cap {cap})")
    finally:
        nv.nvfp4_set_launch_config(0, 0, 0)
    assert nv.nvfp4_get_device_status() == 0


@pytest.mark.parametrize("mode", ["six", "four_over_six_fp16"])
def test_moe_activation_other_modes_every_row(mode):
    x = synth.generate(2, device=DEV)["x"]
    want = oracle_quantize_rows(_u16(x), mode)
    codes, scales, sdec = nv.nvfp4_quantize_rowwise(x, mode)
    assert_same(_np(codes), want["codes"], f"{mode} codes")
    assert_same(_np(scales), want["scales"], f"{mode} block scales")
    assert_same(_np(sdec), want["scale"], f"{mode} row scale")
    assert nv.nvfp4_get_device_status() == 0


def test_moe_activation_residual_every_row():
    x = synth.generate(2, device=DEV)["x"]
    xb = _u16(x)
    rows, cols = xb.shape
    want = [{"codes": np.empty((rows, cols // 2), np.uint8),
             "scales": np.empty((rows, cols // 16), np.uint8),
             "scale": np.empty(rows, np.float32)} for _ in range(2)]

    def one(r):
        a, b = r
        for dst, src in zip(want, oracle.quantize_residual(xb[a:b])):
            for k in dst:
                dst[k][a:b] = src[k]

    _parallel(one, rows)
    got = nv.nvfp4_quantize_residual(x, "four_over_six")
    for part, (g_codes, g_scales, g_scale) in zip(want, got):
        assert_same(_np(g_codes), part["codes"], "residual codes")
        assert_same(_np(g_scales), part["scales"], "residual block scales")
        assert_same(_np(g_scale), part["scale"], "residual row scale")
    assert nv.nvfp4_get_device_status() == 0


def test_moe_activation_guided_every_row():
    """The rollout's record (per-token amax, codes, block scales) is the oracle's; both sides get
    it, and the trainer's values are the rollout's with a few BF16 ulps of noise."""
    x_roll = synth.generate(2, device=DEV)["x"]
    xb = _u16(x_roll)
    rows = xb.shape[0]
    record = oracle_quantize_rows(xb, "four_over_six")
    amax = np.empty(rows, np.float32)

    def amax_rows(r):
        for i in range(*r):
            amax[i] = oracle.amax(xb[i])

    _parallel(amax_rows, rows)
    assert_same(_np(nv.nvfp4_row_amax(x_roll)), amax, "row amax")
    g = torch.Generator(device=DEV).manual_seed(2)
    noise = torch.randn(x_roll.shape, generator=g, device=DEV) * 2.0 ** -7
    x_tr = (x_roll.float() * (1 + noise)).to(torch.bfloat16)
    del noise
    tb = _u16(x_tr)
    want = np.empty_like(record["codes"])

    def guided(r):
        a, b = r
        want[a:b] = oracle.quantize_guided(tb[a:b], amax[a:b], record["codes"][a:b],
                                           record["scales"][a:b])

    _parallel(guided, rows)
    dev = lambda a: torch.from_numpy(a).to(DEV)
    got = nv.nvfp4_quantize_guided(x_tr, dev(amax), dev(record["codes"]), dev(record["scales"]))
    assert_same(_np(got), want, "guided codes")
    assert nv.nvfp4_get_device_status() == 0


def test_expert_grouped_every_row():
    d = synth.generate(3, device=DEV)
    x, offsets = d["x"], d["offsets"]
    want = oracle_quantize_rows(_u16(x), "four_over_six")
    codes, scales, sdec = nv.nvfp4_quantize_rowwise(x, "four_over_six", offsets)
    assert_same(_np(codes), want["codes"], "codes")
    assert_same(_np(scales), want["scales"], "block scales")
    assert_same(_np(sdec), want["scale"], "row scale")
    assert nv.nvfp4_get_device_status() == 0


def test_long_rollout_every_row():
    """131072 x 7168: quantize, dequantize and the fused round trip, every element."""
    x = synth.generate(4, device=DEV)["x"]
    want = oracle_quantize_rows(_u16(x), "four_over_six", want_y=True)
    codes, scales, sdec = nv.nvfp4_quantize_rowwise(x, "four_over_six")
    assert_same(_np(codes), want["codes"], "codes")
    assert_same(_np(scales), want["scales"], "block scales")
    assert_same(_np(sdec), want["scale"], "row scale")
    y = nv.nvfp4_dequantize(codes, scales, sdec, "row")
    assert_same(_u16(y), want["y"], "dequantized y")
    del codes, scales, sdec, y
    codes, scales, sdec, y = nv.nvfp4_fused_roundtrip(x, "row", "four_over_six")
    assert_same(_np(codes), want["codes"], "fused codes")
    assert_same(_np(scales), want["scales"], "fused block scales")
    assert_same(_np(sdec), want["scale"], "fused row scale")
    assert_same(_u16(y), want["y"], "fused y")
    assert nv.nvfp4_get_device_status() == 0
