"""GPU parity: the CUDA library against the CPU oracle, bit for bit, through the C ABI.

Codes, E4M3 block scales, FP32 scales and dequantized BF16 are integer/byte results of a fully
specified FP32 computation, so the bar is exact equality everywhere.  Full-size workloads are run
in the benchmark's launch configuration and checked on sampled rows (the oracle is slow), plus
properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_block_scaled_row_gb300 as nv
from nvfp4_block_scaled_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
F4, SIX, F16 = "four_over_six", "six", "four_over_six_fp16"
OMODE = {F4: oracle.MODE_FOUR_OVER_SIX, SIX: oracle.MODE_SIX, F16: oracle.MODE_FOUR_OVER_SIX_FP16}


@pytest.fixture(scope="module", autouse=True)
def _library():
    nv.library()
    nv.nvfp4_set_launch_config(0, 0, 0)
    nv.nvfp4_get_device_status(clear=True)
    yield
    nv.nvfp4_set_launch_config(0, 0, 0)


def _np(t):
    return t.detach().cpu().numpy()


def _y_u16(y):
    return synth.as_u16(y)


def _assert_equal(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    if got.dtype == np.float32:
        got, want = got.view(np.uint32), want.view(np.uint32)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {i}: "
                             f"gpu={got[i]!r} oracle={want[i]!r}")


def check_rowwise(x, mode=F4, fused=True, dequant=True):
    xb = synth.as_u16(x)
    want = oracle.quantize(xb, OMODE[mode], oracle.SCALE_ROW)
    codes, scales, sdec = nv.nvfp4_quantize_rowwise(x, mode)
    torch.cuda.synchronize()
    _assert_equal(_np(codes), want["codes"], "codes")
    _assert_equal(_np(scales), want["scales"], "block scales")
    _assert_equal(_np(sdec), want["scale"], "row scale")
    ywant = oracle.dequantize(want["codes"], want["scales"], want["scale"], oracle.SCALE_ROW)
    if dequant:
        y = nv.nvfp4_dequantize(codes, scales, sdec, "row")
        _assert_equal(_y_u16(y), ywant, "dequantized y")
    if fused:
        c2, s2, d2, y2 = nv.nvfp4_fused_roundtrip(x, "row", mode)
        _assert_equal(_np(c2), want["codes"], "fused codes")
        _assert_equal(_np(s2), want["scales"], "fused block scales")
        _assert_equal(_np(d2), want["scale"], "fused row scale")
        _assert_equal(_y_u16(y2), ywant, "fused y")
    assert nv.nvfp4_get_device_status() == 0


def check_tensor(x, mode=F4):
    xb = synth.as_u16(x)
    want = oracle.quantize(xb, OMODE[mode], oracle.SCALE_TENSOR)
    ywant = oracle.dequantize(want["codes"], want["scales"], want["scale"], oracle.SCALE_TENSOR)
    codes, scales, ts = nv.nvfp4_quantize_tensor(x, mode)
    _assert_equal(_np(codes), want["codes"], "codes")
    _assert_equal(_np(scales), want["scales"], "block scales")
    _assert_equal(_np(ts), want["scale"], "tensor scale")
    y = nv.nvfp4_dequantize(codes, scales, ts, "tensor")
    _assert_equal(_y_u16(y), ywant, "dequantized y")
    c2, s2, t2, y2 = nv.nvfp4_fused_roundtrip(x, "tensor", mode)
    _assert_equal(_np(c2), want["codes"], "fused codes")
    _assert_equal(_np(s2), want["scales"], "fused block scales")
    _assert_equal(_np(t2), want["scale"], "fused tensor scale")
    _assert_equal(_y_u16(y2), ywant, "fused y")
    amax = nv.nvfp4_tensor_amax(x)
    assert float(amax.item()) == oracle.amax(xb)
    c3, s3, t3 = nv.nvfp4_quantize_tensor_with_amax(x, amax, mode)
    _assert_equal(_np(c3), want["codes"], "with-amax codes")
    _assert_equal(_np(s3), want["scales"], "with-amax block scales")
    _assert_equal(_np(t3), want["scale"], "with-amax tensor scale")
    assert nv.nvfp4_get_device_status() == 0


# ---- the five workloads ------------------------------------------------------------------------

def test_workload0_activation_tiny_full():
    check_rowwise(synth.generate(0, device=DEV)["x"])


@pytest.mark.parametrize("mode", [SIX, F4])
def test_workload1_weight_tensor_scale_full(mode):
    check_tensor(synth.generate(1, device=DEV)["x"], mode)


@pytest.mark.parametrize("index,rows", [(2, 300), (3, 640), (4, 500)])
def test_workloads_small_instances(index, rows):
    d = synth.generate(index, device=DEV, rows=rows)
    check_rowwise(d["x"])
    check_rowwise(d["x"], SIX, fused=False, dequant=False)


def _sample_rows(rows, n=48, seed=0):
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(rows, size=min(n, rows), replace=False).tolist())
    pick |= {0, rows - 1}
    return np.array(sorted(pick))


def _check_sampled(x, codes, scales, sdec, y, rows_idx):
    xs = synth.as_u16(x[torch.as_tensor(rows_idx, device=x.device)])
    want = oracle.quantize(xs, oracle.MODE_FOUR_OVER_SIX, oracle.SCALE_ROW)
    idx = torch.as_tensor(rows_idx, device=x.device)
    _assert_equal(_np(codes[idx]), want["codes"], "sampled codes")
    _assert_equal(_np(scales[idx]), want["scales"], "sampled block scales")
    _assert_equal(_np(sdec[idx]), want["scale"], "sampled row scale")
    if y is not None:
        ywant = oracle.dequantize(want["codes"], want["scales"], want["scale"])
        _assert_equal(_y_u16(y[idx]), ywant, "sampled y")


@pytest.mark.parametrize("index", [2, 3, 4])
def test_full_size_sampled_rows(index):
    """Full-size workloads in the benchmark's launch configuration, checked on sampled rows,
    plus: the separate dequantize equals the fused round trip on every element."""
    d = synth.generate(index, device=DEV)
    x = d["x"]
    rows = x.shape[0]
    codes, scales, sdec, y = nv.nvfp4_fused_roundtrip(x, "row", F4)
    c1, s1, d1 = nv.nvfp4_quantize_rowwise(x, F4, group_offsets=d["offsets"])
    assert torch.equal(c1, codes) and torch.equal(s1, scales) and torch.equal(d1, sdec)
    y2 = nv.nvfp4_dequantize(codes, scales, sdec, "row")
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    picks = _sample_rows(rows, seed=index)
    if index == 4:
        zero_rows = torch.nonzero(x.abs().amax(1) == 0).flatten()[:4].cpu().numpy()
        spike_rows = torch.nonzero(x.abs().amax(1) > 20000).flatten()[:4].cpu().numpy()
        picks = np.unique(np.concatenate([picks, zero_rows, spike_rows]))
        assert float(sdec[torch.as_tensor(zero_rows, device=DEV)].abs().max()) == 0.0
    _check_sampled(x, codes, scales, sdec, y, picks)
    assert nv.nvfp4_get_device_status() == 0


# ---- edge cases --------------------------------------------------------------------------------

def _edge_matrix(rows, cols, seed):
    """Rows that hit the corner cases: exact E2M1/E4M3 ties (small multiples of powers of two),
    zero rows, zero blocks, BF16 subnormals, values near the BF16 maximum, a lone spike,
    negative values that round to zero, and ordinary Gaussian rows."""
    rng = np.random.default_rng(seed)
    x = np.zeros((rows, cols), np.float32)
    for r in range(rows):
        kind = r % 8
        if kind == 0:
            x[r] = rng.integers(-64, 65, cols) * 2.0 ** rng.integers(-4, 4, cols)
        elif kind == 1:
            pass  # zero row
        elif kind == 2:
            x[r] = rng.standard_normal(cols)
            x[r, : min(cols, 16)] = 0.0  # a zero block
        elif kind == 3:
            x[r] = rng.standard_normal(cols) * 2.0 ** -130  # BF16 subnormals
        elif kind == 4:
            x[r] = rng.standard_normal(cols) * 1e37
            x[r, 0] = 3.3e38
        elif kind == 5:
            x[r] = rng.standard_normal(cols) * 1e-3
            x[r, rng.integers(cols)] = 3.0e4
        elif kind == 6:
            x[r] = -rng.uniform(0, 0.01, cols)
            x[r, -1] = 6.0
        else:
            x[r] = rng.standard_normal(cols) * np.exp(rng.uniform(-20, 20))
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.to(DEV)


@pytest.mark.parametrize("cols", [16, 32, 48, 496, 512, 2064, 7168, 7184, 16384, 32768, 65536])
def test_edge_values_and_ragged_widths(cols):
    rows = 3 if cols >= 16384 else 37
    x = _edge_matrix(rows, cols, seed=cols)
    check_rowwise(x)
    check_rowwise(x, SIX, fused=True, dequant=False)
    check_tensor(x[: min(rows, 9)].contiguous(), F4)


def test_block_error_order_blocks():
    """The two blocks whose 4/6 choice only the ascending order of the error chain decides
    (test_oracle_method.chain_order_row), tiled along a 7168-wide row so every lane of a team sees
    them, and alone in a 32-wide row."""
    from test_oracle_method import chain_order_row

    pair = chain_order_row()[0]
    wide = np.tile(pair, 7168 // 32)[None, :]
    for bits in (pair[None, :], wide, np.repeat(wide, 5, axis=0)):
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
        check_rowwise(x)
        check_tensor(x, F4)
    codes, scales, _ = nv.nvfp4_quantize_rowwise(
        torch.from_numpy(pair[None, :].view(np.int16)).view(torch.bfloat16).to(DEV))
    assert list(_np(scales)[0]) == [0x78, 0x7C]


@pytest.mark.parametrize("rows", [1, 2, 7, 31, 33])
def test_few_rows(rows):
    check_rowwise(_edge_matrix(rows, 7168, seed=rows))


def test_zero_rows_is_noop():
    x = torch.empty((0, 7168), dtype=torch.bfloat16, device=DEV)
    codes, scales, sdec = nv.nvfp4_quantize_rowwise(x)
    assert codes.shape == (0, 3584) and scales.shape == (0, 448) and sdec.shape == (0,)
    y = nv.nvfp4_dequantize(codes, scales, sdec)
    assert y.shape == (0, 7168)


# ---- determinism and launch independence -------------------------------------------------------

def test_deterministic_and_launch_shape_independent():
    x = synth.generate(2, device=DEV, rows=1000)["x"]
    base = [t.clone() for t in nv.nvfp4_fused_roundtrip(x)]
    shapes = [(1, 1, 0), (1, 2, 1), (3, 1, 5), (8, 2, 0), (2, 4, 17), (0, 0, 3), (7, 3, 0)]
    try:
        for w, s, c in shapes:
            nv.nvfp4_set_launch_config(w, s, c)
            out = nv.nvfp4_fused_roundtrip(x)
            for a, b in zip(base, out):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (w, s, c)
            t = nv.nvfp4_quantize_tensor(x)
            assert torch.equal(t[0], nv.nvfp4_quantize_tensor(x)[0])
    finally:
        nv.nvfp4_set_launch_config(0, 0, 0)
    again = nv.nvfp4_fused_roundtrip(x)
    for a, b in zip(base, again):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_batch_independence_on_gpu():
    x = synth.generate(3, device=DEV, rows=700)["x"]
    codes, scales, sdec = nv.nvfp4_quantize_rowwise(x)
    perm = torch.randperm(x.shape[0], device=DEV, generator=torch.Generator(DEV).manual_seed(1))
    c2, s2, d2 = nv.nvfp4_quantize_rowwise(x[perm].contiguous())
    assert torch.equal(c2, codes[perm]) and torch.equal(s2, scales[perm])
    assert torch.equal(d2, sdec[perm])
    c3, s3, d3 = nv.nvfp4_quantize_rowwise(x[:123].contiguous())
    assert torch.equal(c3, codes[:123]) and torch.equal(d3, sdec[:123])


def test_streams_are_honoured():
    x = synth.generate(2, device=DEV, rows=512)["x"]
    ref = nv.nvfp4_fused_roundtrip(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = nv.nvfp4_fused_roundtrip(x, stream=s)
    s.synchronize()
    for a, b in zip(ref, out):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


# ---- device-side error reporting ---------------------------------------------------------------

def test_group_offsets_validation():
    d = synth.generate(3, device=DEV, rows=640)
    x, off = d["x"], d["offsets"]
    nv.nvfp4_quantize_rowwise(x, group_offsets=off)
    assert nv.nvfp4_get_device_status() == 0
    bad = off.clone()
    bad[5], bad[6] = off[6] + 1, off[5]  # not monotone
    nv.nvfp4_quantize_rowwise(x, group_offsets=bad)
    assert nv.nvfp4_get_device_status() == 6
    short = off.clone()
    short[-1] = x.shape[0] - 1  # does not end at rows
    nv.nvfp4_quantize_rowwise(x, group_offsets=short)
    assert nv.nvfp4_get_device_status() == 6
    assert nv.nvfp4_get_device_status() == 0  # cleared by the read


def test_bounded_wait_reports_timeout():
    nv.nvfp4_get_device_status(clear=True)
    nv.nvfp4_selftest_wait_timeout(200_000)  # 0.2 ms on a barrier nobody arrives on
    assert nv.nvfp4_get_device_status() == 5
    # The context is still healthy afterwards.
    check_rowwise(synth.generate(0, device=DEV, rows=16)["x"])


@pytest.mark.parametrize("cols,op", [(7168, "rowwise"), (7168, "fused"), (7168, "tensor"),
                                     (7168, "residual"), (2048, "rowwise"), (32768, "rowwise"),
                                     (65536, "rowwise"), (7168, "fused_units")])
def test_quantize_ring_timeout_path(cols, op):
    """The quantize kernel's own failure branches: with one row's copies withheld, the warps that
    own it give up after 1 ms, record NVFP4_ERR_TIMEOUT, drain their copies still in flight and
    return (a team of several warps -- 2 for 7168-wide rows, 8 for 32768, 16 for 65536 -- leaves
    together behind its barrier); the next ordinary call on the same context is bit-exact.
    fused_units: 2435 rows, so the withheld row sits in a work unit that a running CTA took over
    from one that had not started, and the CTAs still waiting for work-unit answers after the
    failing team left give up in bounded time too; the next call matches a clean call before it
    (whose rows the other tests check against the oracle)."""
    if op == "fused_units":
        x = synth.generate(2, device=DEV, rows=8 * 152 * 2 + 3)["x"]
        base = [t.clone() for t in nv.nvfp4_fused_roundtrip(x, "row")]
        nv.nvfp4_get_device_status(clear=True)
        nv.nvfp4_selftest_withhold_row(2000, 1_000_000)
        try:
            nv.nvfp4_fused_roundtrip(x, "row")
            torch.cuda.synchronize()
        finally:
            nv.nvfp4_selftest_withhold_row(-1, 0)
        assert nv.nvfp4_get_device_status(clear=True) == 5  # NVFP4_ERR_TIMEOUT
        again = nv.nvfp4_fused_roundtrip(x, "row")
        for a, b in zip(base, again):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
        assert nv.nvfp4_get_device_status() == 0
        return
    if cols == 2048:
        x = synth.generate(0, device=DEV, rows=96)["x"]
    elif cols == 7168:
        x = synth.generate(2, device=DEV, rows=96)["x"]
    else:
        x = _edge_matrix(12, cols, seed=5)
    nv.nvfp4_get_device_status(clear=True)
    nv.nvfp4_selftest_withhold_row(3, 1_000_000)
    try:
        if op == "rowwise":
            nv.nvfp4_quantize_rowwise(x)
        elif op == "fused":
            nv.nvfp4_fused_roundtrip(x, "row")
        elif op == "tensor":
            nv.nvfp4_quantize_tensor(x)
        else:
            nv.nvfp4_quantize_residual(x)
        torch.cuda.synchronize()
    finally:
        nv.nvfp4_selftest_withhold_row(-1, 0)
    assert nv.nvfp4_get_device_status(clear=True) == 5  # NVFP4_ERR_TIMEOUT
    check_rowwise(x, F4, fused=True, dequant=False)
    if op == "tensor":
        check_tensor(x, F4)
    if op == "residual":
        check_residual(x)


def test_host_validation_errors():
    x = synth.generate(0, device=DEV, rows=4)["x"]
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_quantize_rowwise(x[:, :24].contiguous())
    assert e.value.status == 2
    with pytest.raises(ValueError):
        nv.nvfp4_quantize_rowwise(x.cpu())
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_quantize_rowwise(torch.empty((4, 65536 + 16), dtype=torch.bfloat16, device=DEV))
    assert e.value.status == 2


def test_sharded_tensor_helper_on_one_rank():
    from nvfp4_block_scaled_row_gb300 import distributed as D

    x = synth.generate(1, device=DEV, rows=256)["x"]
    want = nv.nvfp4_quantize_tensor(x)
    got = D.quantize_tensor_sharded(x)
    for a, b in zip(want, got):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_host_streamed_roundtrip_matches_device_call():
    """Host-resident input streamed in chunks (several chunks and a ragged last one) gives the
    device call's outputs exactly, for both modes."""
    x = synth.generate(2, device=DEV, rows=5000)["x"]  # three ~32 MB chunks, the last ragged
    xh = x.cpu().pin_memory()
    for mode in (F4, SIX):
        want = nv.nvfp4_fused_roundtrip(x, "row", mode)
        got = nv.nvfp4_fused_roundtrip_host(xh, mode)
        torch.cuda.current_stream().synchronize()
        for a, b in zip(want, got):
            assert torch.equal(a.cpu().view(torch.uint8), b.view(torch.uint8))
    # pageable host memory also works (serialized copies)
    got = nv.nvfp4_fused_roundtrip_host(x[:300].cpu())
    torch.cuda.current_stream().synchronize()
    assert torch.equal(got[0], nv.nvfp4_fused_roundtrip(x[:300].contiguous())[0].cpu())
    assert nv.nvfp4_get_device_status() == 0


def test_host_streamed_roundtrip_concurrent_callers():
    """Two host threads streaming different matrices on their own streams at the same time (the
    internal streams are shared per device) each get their own device call's outputs."""
    import threading

    xs = [synth.generate(i, device=DEV, rows=3000)["x"] for i in (2, 4)]
    hosts = [x.cpu().pin_memory() for x in xs]
    wants = [nv.nvfp4_fused_roundtrip(x) for x in xs]
    torch.cuda.synchronize()
    results, errors = [None, None], []

    def run(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            outs = []
            for _ in range(3):
                outs = nv.nvfp4_fused_roundtrip_host(hosts[i], stream=st)
            st.synchronize()
            results[i] = outs
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in (0, 1)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for want, got in zip(wants, results):
        for a, b in zip(want, got):
            assert torch.equal(a.cpu().view(torch.uint8), b.view(torch.uint8))
    assert nv.nvfp4_get_device_status() == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_against_oracle(seed):
    """Random widths (any multiple of 16 up to 8192), row counts and modes, row and tensor scale,
    on the edge-case value mix."""
    rng = np.random.default_rng(100 + seed)
    for _ in range(4):
        cols = 16 * int(rng.integers(1, 513))
        rows = int(rng.integers(1, 97))
        mode = (F4, SIX, F16)[int(rng.integers(0, 3))]
        x = _edge_matrix(rows, cols, seed=int(rng.integers(1 << 30)))
        check_rowwise(x, mode)
        check_tensor(x, mode)


def check_residual(x, mode=F4, rows_idx=None):
    xs = x if rows_idx is None else x[torch.as_tensor(rows_idx, device=x.device)]
    want_m, want_r = oracle.quantize_residual(synth.as_u16(xs), OMODE[mode])
    (c, s, d), (rc, rs, rd) = nv.nvfp4_quantize_residual(x, mode)
    if rows_idx is not None:
        idx = torch.as_tensor(rows_idx, device=x.device)
        c, s, d, rc, rs, rd = (t[idx] for t in (c, s, d, rc, rs, rd))
    for got, want, what in ((c, want_m["codes"], "codes"), (s, want_m["scales"], "scales"),
                            (d, want_m["scale"], "row scale"), (rc, want_r["codes"], "res codes"),
                            (rs, want_r["scales"], "res scales"),
                            (rd, want_r["scale"], "res row scale")):
        _assert_equal(_np(got), want, what)
    assert nv.nvfp4_get_device_status() == 0


@pytest.mark.parametrize("index,rows", [(0, None), (2, 300), (3, 640), (4, 500)])
def test_residual_workloads(index, rows):
    x = synth.generate(index, device=DEV, rows=rows)["x"]
    check_residual(x)
    check_residual(x, SIX)


@pytest.mark.parametrize("cols", [16, 48, 2064, 7168, 7184, 32768, 65536])
def test_residual_edge_values(cols):
    check_residual(_edge_matrix(3 if cols >= 16384 else 21, cols, seed=cols + 1))


def test_residual_full_size_sampled():
    x = synth.generate(2, device=DEV)["x"]
    check_residual(x, F4, _sample_rows(x.shape[0], n=32, seed=7))



def _perturbed(x, seed):
    """The training engine's view of the rollout's activations: a few BF16 ulps of noise."""
    g = torch.Generator(device=x.device).manual_seed(seed)
    noise = torch.randn(x.shape, generator=g, device=x.device) * 2.0 ** -7
    return (x.float() * (1 + noise)).to(torch.bfloat16)


def _oracle_record(x_roll):
    """The rollout's record as the oracle computes it: per-token amax, codes and block scales
    (numpy, for the oracle) and the same arrays on the device (for the library)."""
    xb = synth.as_u16(x_roll)
    amax = np.array([oracle.amax(xb[r]) for r in range(xb.shape[0])], np.float32)
    q = oracle.quantize(xb, oracle.MODE_FOUR_OVER_SIX, oracle.SCALE_ROW)
    host = (amax, q["codes"], q["scales"])
    return host, tuple(torch.from_numpy(a).to(DEV) for a in host)


@pytest.mark.parametrize("index,rows", [(0, None), (2, 256), (4, 300)])
def test_guided_rounding_matches_oracle(index, rows):
    x_roll = synth.generate(index, device=DEV, rows=rows)["x"]
    (amax_h, codes_h, scales_h), (amax, codes, scales) = _oracle_record(x_roll)
    _assert_equal(_np(nv.nvfp4_row_amax(x_roll)), amax_h, "row amax")
    same = nv.nvfp4_quantize_guided(x_roll, amax, codes, scales)
    assert torch.equal(same, codes)  # trainer == rollout -> the rollout's codes
    x_tr = _perturbed(x_roll, index)
    got = nv.nvfp4_quantize_guided(x_tr, amax, codes, scales)
    want = oracle.quantize_guided(synth.as_u16(x_tr), amax_h, codes_h, scales_h)
    _assert_equal(_np(got), want, "guided codes")
    own = nv.nvfp4_quantize_guided(x_tr, amax, got, scales)  # idempotent on its own output
    assert torch.equal(own, got)
    assert nv.nvfp4_get_device_status() == 0


def test_guided_ring_timeout_path():
    """The staged guided encoder's failure branch: with one row's copies withheld, the warp whose
    units include it gives up after 1 ms, records NVFP4_ERR_TIMEOUT, drains its copies still in
    flight and returns; the next ordinary call on the same context matches the oracle."""
    x_roll = synth.generate(2, device=DEV, rows=96)["x"]
    (amax_h, codes_h, scales_h), (amax, codes, scales) = _oracle_record(x_roll)
    x_tr = _perturbed(x_roll, 2)
    nv.nvfp4_get_device_status(clear=True)
    nv.nvfp4_selftest_withhold_row(5, 1_000_000)
    try:
        nv.nvfp4_quantize_guided(x_tr, amax, codes, scales)
        torch.cuda.synchronize()
    finally:
        nv.nvfp4_selftest_withhold_row(-1, 0)
    assert nv.nvfp4_get_device_status(clear=True) == 5  # NVFP4_ERR_TIMEOUT
    got = nv.nvfp4_quantize_guided(x_tr, amax, codes, scales)
    want = oracle.quantize_guided(synth.as_u16(x_tr), amax_h, codes_h, scales_h)
    _assert_equal(_np(got), want, "guided codes after the timeout")
    assert nv.nvfp4_get_device_status() == 0


@pytest.mark.parametrize("rows,cols", [(16, 16), (16, 48), (16, 7184), (1, 1024), (77, 1024),
                                       (5, 3072), (16, 4096)])
def test_guided_rounding_edge_values(rows, cols):
    """Edge values through both guided kernels: widths that are whole 1024-element units take the
    staged one (one unit, fewer units than warps, several units per row), the others the direct one."""
    x_roll = _edge_matrix(rows, cols, seed=cols + 3 + rows)
    (amax_h, codes_h, scales_h), (amax, codes, scales) = _oracle_record(x_roll)
    x_tr = _perturbed(x_roll, cols)
    got = nv.nvfp4_quantize_guided(x_tr, amax, codes, scales)
    want = oracle.quantize_guided(synth.as_u16(x_tr), amax_h, codes_h, scales_h)
    _assert_equal(_np(got), want, "guided codes (edge)")



@pytest.mark.parametrize("index,rows", [(0, None), (2, 300), (3, 640), (4, 500)])
def test_fp16_selector_mode(index, rows):
    """The FP16 reading of the 4/6 fast path is bit-exact against its oracle statement too."""
    x = synth.generate(index, device=DEV, rows=rows)["x"]
    check_rowwise(x, F16)
    check_residual(x, F16)
    if index == 0:
        check_tensor(x, F16)


def test_fp16_selector_edge_values():
    x = _edge_matrix(37, 7184, seed=11)
    check_rowwise(x, F16)
    check_tensor(x[:9].contiguous(), F16)



def _swizzle_reference(scales):
    """The tiled layout written out plainly: tile (r // 128, c // 4), byte
    (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4 inside it, zero padding."""
    rows, sc = scales.shape
    tr, tc = -(-rows // 128), -(-sc // 4)
    out = np.zeros(tr * tc * 512, np.uint8)
    for r in range(rows):
        for c in range(sc):
            tile = (r // 128) * tc + c // 4
            out[tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4] = scales[r, c]
    return out


@pytest.mark.parametrize("rows,cols", [(1, 16), (130, 7168), (256, 2048), (77, 1040)])
def test_swizzle_block_scales(rows, cols):
    x = _edge_matrix(rows, cols, seed=rows)
    _, scales, _ = nv.nvfp4_quantize_rowwise(x)
    got = nv.nvfp4_swizzle_block_scales(scales, cols)
    assert np.array_equal(_np(got), _swizzle_reference(_np(scales)))


def _oracle_operand(x, kind):
    """An operand quantized by the oracle (4/6; per-token for x, per-tensor for w): its host
    arrays for the float64 reference and the same arrays on the device for the library."""
    q = oracle.quantize(synth.as_u16(x), oracle.MODE_FOUR_OVER_SIX,
                        oracle.SCALE_ROW if kind == "row" else oracle.SCALE_TENSOR)
    return q, tuple(torch.from_numpy(q[k]).to(DEV) for k in ("codes", "scales", "scale"))


def _gemm_check(got, X, W, k):
    """got (float64) against the float64 product X . W^T of the exactly dequantized operands:
    within the BF16 output rounding (2^-9, plus the two FP32 epilogue roundings) and the FP32
    accumulation over k terms (at most k * 2^-24 of the magnitude sum)."""
    ref = X @ W.T
    mag = np.abs(X) @ np.abs(W).T
    bound = 2.0 ** -8 * np.abs(ref) + k * 2.0 ** -24 * mag + 1e-30
    bad = np.abs(got - ref) > bound
    worst = (np.abs(got - ref) / (np.abs(ref) + k * 2.0 ** -24 * mag + 1e-30)).max()
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outputs off; first at "
                           f"{tuple(np.argwhere(bad)[0])}; worst relative error {worst:.3e}")
    return worst


@pytest.mark.parametrize("m,n,k", [(128, 128, 256), (256, 256, 2048), (300, 144, 320),
                                   (512, 384, 7168), (640, 272, 768)])
def test_gemm_nt_matches_float64_product(m, n, k):
    """y = x . Q(w) on the tensor cores against the float64 product of the exactly dequantized
    operands (decoded independently of the library).  Both operands are quantized by the oracle;
    the shapes cover one tile, ragged row and column tiles and a K that ends mid-stage."""
    from indep import exact_dequant

    x = synth.generate(2, device=DEV, rows=m)["x"][:, :k].contiguous()
    w = synth.generate(1, device=DEV, rows=n)["x"][:, :k].contiguous()
    qx, (xc, xs, xd) = _oracle_operand(x, "row")
    qw, (wc, ws, wd) = _oracle_operand(w, "tensor")
    y = nv.nvfp4_gemm_nt(xc, nv.nvfp4_swizzle_block_scales(xs, k), xd,
                         wc, nv.nvfp4_swizzle_block_scales(ws, k), wd)
    worst = _gemm_check(y.float().cpu().numpy().astype(np.float64), exact_dequant(qx, k),
                        exact_dequant(qw, k), k)
    print(f"gemm {m}x{n}x{k}: worst relative error {worst:.3e}")
    assert nv.nvfp4_get_device_status() == 0


def test_gemm_nt_full_size_sampled_rows():
    """The benchmark's product, 16384 x 2048 x 7168 (MoE activations times one expert's weight),
    in its launch configuration; 64 sampled rows of y against the float64 product."""
    from indep import exact_dequant

    k = 7168
    x = synth.generate(2, device=DEV)["x"]
    w = synth.generate(1, device=DEV)["x"]
    qw, (wc, ws, wd) = _oracle_operand(w, "tensor")
    xc, xs, xd = nv.nvfp4_quantize_rowwise(x)
    y = nv.nvfp4_gemm_nt(xc, nv.nvfp4_swizzle_block_scales(xs, k), xd,
                         wc, nv.nvfp4_swizzle_block_scales(ws, k), wd)
    rows = _sample_rows(x.shape[0], n=62, seed=3)
    qx = oracle.quantize(synth.as_u16(x[torch.as_tensor(rows, device=DEV)]),
                         oracle.MODE_FOUR_OVER_SIX, oracle.SCALE_ROW)
    got = y[torch.as_tensor(rows, device=DEV)].float().cpu().numpy().astype(np.float64)
    _gemm_check(got, exact_dequant(qx, k), exact_dequant(qw, k), k)
    assert nv.nvfp4_get_device_status() == 0


def test_device_calls_capture_into_cuda_graphs():
    """Every device entry point can be captured into a CUDA graph (no host synchronisation or
    allocation inside the library) and the replay reproduces the eager outputs."""
    x = synth.generate(2, device=DEV, rows=700)["x"]
    w = synth.generate(1, device=DEV, rows=256)["x"]
    eager = {
        "row": nv.nvfp4_quantize_rowwise(x),
        "fused": nv.nvfp4_fused_roundtrip(x),
        "fused_t": nv.nvfp4_fused_roundtrip(x, "tensor"),
        "tensor": nv.nvfp4_quantize_tensor(w),
        "residual": sum(nv.nvfp4_quantize_residual(x), ()),
    }
    amax = nv.nvfp4_row_amax(x)
    eager["guided"] = (nv.nvfp4_quantize_guided(x, amax, eager["row"][0], eager["row"][1]),)
    eager["deq"] = (nv.nvfp4_dequantize(*eager["row"]),)
    torch.cuda.synchronize()
    outs = {k: tuple(torch.empty_like(t) for t in v) for k, v in eager.items()}
    ws = [torch.empty(nv.nvfp4_tensor_workspace_bytes(), dtype=torch.uint8, device=DEV)
          for _ in range(2)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        nv.nvfp4_quantize_rowwise(x, "four_over_six", None, *outs["row"])
        nv.nvfp4_fused_roundtrip(x, "row", "four_over_six", *outs["fused"])
        nv.nvfp4_fused_roundtrip(x, "tensor", "four_over_six", *outs["fused_t"], ws[0])
        nv.nvfp4_quantize_tensor(w, "four_over_six", *outs["tensor"], ws[1])
        nv.nvfp4_dequantize(*eager["row"], "row", outs["deq"][0])
        nv.nvfp4_quantize_guided(x, amax, eager["row"][0], eager["row"][1], "four_over_six",
                                 outs["guided"][0])
        outs["residual"] = sum(nv.nvfp4_quantize_residual(x), ())  # graph-pool outputs
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for k in ("row", "fused", "fused_t", "tensor", "deq", "guided", "residual"):
        for a, b in zip(eager[k], outs[k]):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), k
    assert nv.nvfp4_get_device_status() == 0


def test_programmatic_launch_waits_for_the_producer():
    """Each library kernel starts as a programmatic dependent of the previous kernel on the stream;
    it must still see everything that kernel wrote.  A torch kernel rewrites x in place right
    before every call (eagerly and inside a CUDA graph); each call's outputs must match a call on
    an unshared copy of the new x."""
    x = synth.generate(2, device=DEV, rows=3000)["x"]
    want = [nv.nvfp4_fused_roundtrip(x.neg() if i % 2 == 0 else x.clone()) for i in range(2)]
    want_q = [nv.nvfp4_quantize_rowwise(x.neg() if i % 2 == 0 else x.clone()) for i in range(2)]
    torch.cuda.synchronize()
    outs = [tuple(torch.empty_like(t) for t in w) for w in want]
    outs_q = [tuple(torch.empty_like(t) for t in w) for w in want_q]
    for step in range(6):
        x.neg_()  # the producer: rewrites x just before the consumer launch
        nv.nvfp4_fused_roundtrip(x, "row", "four_over_six", *outs[step % 2])
        nv.nvfp4_quantize_rowwise(x, "four_over_six", None, *outs_q[step % 2])
        nv.nvfp4_dequantize(*outs_q[step % 2], "row", outs[step % 2][3])  # reads the line above
    torch.cuda.synchronize()
    for w, o in zip(want, outs):
        for a, b in zip(w, o):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    for w, o in zip(want_q, outs_q):
        for a, b in zip(w, o):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    # the same inside a captured graph
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        x.neg_()
        nv.nvfp4_fused_roundtrip(x, "row", "four_over_six", *outs[0])
        x.neg_()
        nv.nvfp4_fused_roundtrip(x, "row", "four_over_six", *outs[1])
    g.replay()
    torch.cuda.synchronize()
    for w, o in zip(want, outs):
        for a, b in zip(w, o):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert nv.nvfp4_get_device_status() == 0


@pytest.mark.parametrize("cols", [7168, 2048, 528])
def test_signed_zero_rows(cols):
    """Rows whose amax is zero hold only +0 and -0: codes carry each element's sign, scales and
    S_dec are zero and y reproduces x bit for bit (row and tensor scale, fused and separate)."""
    rng = np.random.default_rng(cols)
    rows = 40
    bits = np.where(rng.random((rows, cols)) < 0.5, 0x8000, 0x0000).astype(np.uint16)
    bits[3] = 0x8000  # an all -0 row
    bits[4] = 0       # an all +0 row
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    x[5:9] = synth.generate(2, device=DEV, rows=4)["x"][:, :cols]  # some ordinary rows among them
    check_rowwise(x)
    check_rowwise(x, SIX)
    c, s, d, y = nv.nvfp4_fused_roundtrip(x)
    assert torch.equal(y[:5].view(torch.int16), x[:5].view(torch.int16))
    zero_only = x[:5].contiguous()
    check_tensor(zero_only)


def test_concurrent_host_threads_device_calls():
    """Host threads calling the device entry points at once, each on its own stream, with launch
    shapes seen for the first time (the per-device launch caches fill concurrently): every
    output equals the single-threaded result."""
    import threading

    inputs = [synth.generate(2, device=DEV, rows=r)["x"] for r in (97, 513, 1500, 2222)]
    wants = [nv.nvfp4_fused_roundtrip(x) for x in inputs]
    wants_t = [nv.nvfp4_quantize_tensor(x) for x in inputs]
    torch.cuda.synchronize()
    errors = []

    def run(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            x = inputs[i]
            with torch.cuda.stream(st):
                for _ in range(20):
                    got = nv.nvfp4_fused_roundtrip(x)
                    got_t = nv.nvfp4_quantize_tensor(x)
            st.synchronize()
            for a, b in zip(wants[i] + wants_t[i], got + got_t):
                if not torch.equal(a.view(torch.uint8), b.view(torch.uint8)):
                    errors.append(i)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(inputs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert nv.nvfp4_get_device_status() == 0
