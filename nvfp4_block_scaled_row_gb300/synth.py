"""Seeded synthetic inputs for the five workloads the quantizer is measured and checked on.

This module only draws numbers; it holds none of the quantizer's arithmetic.  The same tensor
(generated once, then copied where needed) feeds both the CUDA library and the CPU oracle.

Every workload is drawn with ``torch.Generator`` on the device that will hold it, seeded with
``1000 + index``.  Values are drawn in FP32 and rounded to BF16 by ``Tensor.to``.  A CPU draw and
a CUDA draw with the same seed give different (equally valid) samples, so parity checks always
compare both implementations on one drawn tensor.  Large workloads are drawn in fixed-size row
chunks so device memory stays bounded.

Workloads (hidden sizes follow DeepSeek-V3-style MoE layers):
  0 activation_tiny    X [256 x 2048], N(0,1), 4 random channels x50; row scale, 4/6,
                       quantize then dequantize.
  1 weight_expert_up   W [2048 x 7168], N(0, 0.02^2), round(0.1% of entries) x20; tensor scale,
                       modes six and four_over_six, then dequantize.
  2 moe_activation     X [16384 x 7168], row r ~ N(0, sigma_r^2), sigma_r log-uniform on
                       [0.1, 10], 16 fixed outlier channels x100; row scale, 4/6, fused round trip.
  3 expert_grouped     64 experts, Poisson(512) tokens each, concatenated [~32768 x 7168] with
                       int32 offsets[65]; N(0,1) with Student-t(nu=3) rows on 5% of tokens;
                       row scale, 4/6 quantize.
  4 long_rollout       X [131072 x 7168], Student-t(nu=4), 10% all-zero rows, 1% of rows with a
                       single +-3e4 spike; row scale, 4/6, quantize then dequantize (and fused).
"""
from dataclasses import dataclass

import torch

SEED_BASE = 1000
CHUNK_ROWS = 8192


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    rows: int          # nominal row count (workload 3: the expected total of the Poisson draw)
    cols: int
    scale_kind: str    # "row" or "tensor"
    modes: tuple       # quantizer modes the workload runs
    ops: tuple         # "quantize", "dequantize", "roundtrip"
    summary: str


WORKLOADS = (
    Workload(0, "activation_tiny", 256, 2048, "row", ("four_over_six",),
             ("quantize", "dequantize"),
             "X bf16 [256 x 2048], N(0,1), 4 channels x50; per-token scale, 4/6, then dequantize"),
    Workload(1, "weight_expert_up", 2048, 7168, "tensor", ("six", "four_over_six"),
             ("quantize", "dequantize"),
             "W bf16 [2048 x 7168], N(0,0.02^2), 0.1% entries x20; per-tensor scale, six and 4/6"),
    Workload(2, "moe_activation", 16384, 7168, "row", ("four_over_six",),
             ("roundtrip",),
             "X bf16 [16384 x 7168], sigma_r log-uniform [0.1,10], 16 outlier channels x100; "
             "per-token scale, 4/6, fused quantize->dequantize"),
    Workload(3, "expert_grouped", 32768, 7168, "row", ("four_over_six",),
             ("quantize",),
             "64 experts x Poisson(512) tokens, bf16 [~32768 x 7168] + int32 offsets[65], "
             "N(0,1) with 5% Student-t(3) rows; per-token scale, 4/6"),
    Workload(4, "long_rollout", 131072, 7168, "row", ("four_over_six",),
             ("quantize", "dequantize", "roundtrip"),
             "X bf16 [131072 x 7168], Student-t(4), 10% zero rows, 1% rows with one +-3e4 spike; "
             "per-token scale, 4/6"),
)


def workload(index_or_name):
    for w in WORKLOADS:
        if index_or_name in (w.index, w.name):
            return w
    raise KeyError(index_or_name)


def _generator(index, device):
    g = torch.Generator(device=device)
    g.manual_seed(SEED_BASE + index)
    return g


def _student_t(shape, nu, g, device):
    """Student-t(nu) for integer nu: Z / sqrt(chi2_nu / nu), chi2_nu a sum of nu squared normals."""
    z = torch.randn(shape, generator=g, device=device)
    chi2 = torch.zeros(shape, device=device)
    for _ in range(nu):
        chi2 += torch.randn(shape, generator=g, device=device).square()
    return z / torch.sqrt(chi2 / nu)


def _chunks(rows):
    start = 0
    while start < rows:
        stop = min(rows, start + CHUNK_ROWS)
        yield start, stop
        start = stop


def generate(index, device="cpu", rows=None):
    """Draw workload ``index`` on ``device``.

    ``rows`` overrides the row count (workload 3: the expected total, i.e. 64 x the Poisson mean)
    for smaller instances with the same recipe.  Returns a dict with ``x`` (bf16 [rows, cols]) and
    ``offsets`` (int32 [65] on ``device`` for workload 3, else None).
    """
    w = workload(index)
    device = torch.device(device)
    g = _generator(w.index, device)
    cols = w.cols
    nominal = w.rows if rows is None else int(rows)
    offsets = None

    if w.index == 0:
        x = torch.randn((nominal, cols), generator=g, device=device)
        channels = torch.randperm(cols, generator=g, device=device)[:4]
        x[:, channels] *= 50.0
        x = x.to(torch.bfloat16)

    elif w.index == 1:
        n = nominal * cols
        x = torch.randn((nominal, cols), generator=g, device=device) * 0.02
        k = int(round(0.001 * n))
        picks = torch.randperm(n, generator=g, device=device)[:k]
        x.view(-1)[picks] *= 20.0
        x = x.to(torch.bfloat16)

    elif w.index == 2:
        log_sigma = torch.empty(nominal, device=device).uniform_(-1.0, 1.0, generator=g)
        sigma = torch.pow(10.0, log_sigma)
        channels = torch.randperm(cols, generator=g, device=device)[:16]
        x = torch.empty((nominal, cols), dtype=torch.bfloat16, device=device)
        for a, b in _chunks(nominal):
            part = torch.randn((b - a, cols), generator=g, device=device) * sigma[a:b, None]
            part[:, channels] *= 100.0
            x[a:b] = part.to(torch.bfloat16)

    elif w.index == 3:
        experts = 64
        mean = nominal / experts
        # Poisson counts are drawn on the CPU so the group sizes do not depend on the device.
        gc = torch.Generator().manual_seed(SEED_BASE + w.index)
        counts = torch.poisson(torch.full((experts,), float(mean)), generator=gc).to(torch.int64)
        total = int(counts.sum())
        offs = torch.zeros(experts + 1, dtype=torch.int64)
        offs[1:] = torch.cumsum(counts, 0)
        offsets = offs.to(torch.int32).to(device)
        heavy = torch.rand(total, generator=g, device=device) < 0.05
        x = torch.empty((total, cols), dtype=torch.bfloat16, device=device)
        for a, b in _chunks(total):
            part = torch.randn((b - a, cols), generator=g, device=device)
            t3 = _student_t((b - a, cols), 3, g, device)
            part = torch.where(heavy[a:b, None], t3, part)
            x[a:b] = part.to(torch.bfloat16)

    elif w.index == 4:
        x = torch.empty((nominal, cols), dtype=torch.bfloat16, device=device)
        for a, b in _chunks(nominal):
            x[a:b] = _student_t((b - a, cols), 4, g, device).to(torch.bfloat16)
        order = torch.randperm(nominal, generator=g, device=device)
        n_zero = int(round(0.10 * nominal))
        n_spike = int(round(0.01 * nominal))
        zero_rows = order[:n_zero]
        spike_rows = order[n_zero:n_zero + n_spike]
        x[zero_rows] = 0
        spike_cols = torch.randint(0, cols, (n_spike,), generator=g, device=device)
        signs = torch.randint(0, 2, (n_spike,), generator=g, device=device) * 2 - 1
        x[spike_rows, spike_cols] = (signs.to(torch.float32) * 3.0e4).to(torch.bfloat16)

    else:  # pragma: no cover
        raise KeyError(index)

    return {"x": x.contiguous(), "offsets": offsets}


def as_u16(x):
    """Host numpy uint16 view of a bf16 tensor's bit patterns (what the oracle consumes)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
