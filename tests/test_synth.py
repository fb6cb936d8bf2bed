"""The seeded workload generators: deterministic, right shapes, right structure."""
import torch

from nvfp4_block_scaled_row_gb300 import synth


def test_deterministic_per_seed():
    for i, rows in ((0, None), (2, 32), (4, 64)):
        a = synth.generate(i, rows=rows)["x"]
        b = synth.generate(i, rows=rows)["x"]
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shapes_and_dtypes():
    for w in synth.WORKLOADS:
        rows = 64 if w.index != 3 else 640
        d = synth.generate(w.index, rows=rows if w.index else None)
        x = d["x"]
        assert x.dtype == torch.bfloat16 and x.is_contiguous() and x.shape[1] == w.cols
        assert w.cols % 16 == 0


def test_workload0_outlier_channels():
    x = synth.generate(0)["x"].float()
    col_max = x.abs().amax(0)
    assert int((col_max > 40).sum()) == 4


def test_workload1_outlier_count():
    x = synth.generate(1, rows=64)["x"].float()
    n = x.numel()
    assert int((x.abs() > 0.2).sum()) >= round(0.001 * n) * 0.5
    assert x.abs().max() < 3.0


def test_workload3_offsets():
    d = synth.generate(3, rows=1280)
    off = d["offsets"]
    assert off.dtype == torch.int32 and off.numel() == 65
    assert int(off[0]) == 0 and int(off[-1]) == d["x"].shape[0]
    assert bool((off[1:] >= off[:-1]).all())


def test_workload4_zero_rows_and_spikes():
    x = synth.generate(4, rows=1000)["x"].float()
    assert int((x.abs().amax(1) == 0).sum()) == 100
    assert int((x.abs() > 29000).sum()) == 10
