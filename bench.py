#!/usr/bin/env python
"""Throughput of the GB300 NVFP4 4/6 quantizer, as one JSON line.

Headline workload: the long-rollout batch, X bf16 [131072 x 7168] (Student-t(4) entries, 10%
all-zero rows, 1% rows with one +-3e4 spike), per-token FP32 scale, Four-Over-Six block scales,
fused quantize -> dequantize round trip (codes, E4M3 scales, row scales and BF16 y), i.e. one
launch of nvfp4_fused_roundtrip per step: the largest of the five workloads.  Inputs are drawn
on the device (seeded) and stay resident; the 1.88 GB input exceeds the 129 MB L2, so no step
reads the previous step's data from L2.

  value     algorithmic HBM bytes (2 B in + 0.5625 B codes/scales + 2 B y per element + 4 B per
            row) per step / device time per step, summed over ranks, in GB/s; the K timed steps
            are captured once into a CUDA graph and replayed (no host launch overhead)
  e2e       the same metric through the public API with pinned host buffers: every step copies
            x host->device, runs the call, and copies all outputs back
  roofline  the fused kernel's achieved GB/s against the measured HBM copy bandwidth
  cpu_baseline  the CPU oracle on a bounded sample of the same rows (all host cores, and one)
  also      kernel-only GB/s of the other workloads and operations
  cpu_baselines the CPU oracle on a bounded sample of every workload (all host cores, and one)

--impl reference times the CPU oracle instead (the only reference this method has).
Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no collective on the path).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = 4
METRIC = "NVFP4 4/6 quantize GB/s and elem/s, fraction of GB300 HBM peak"
L2_BYTES = 129 * 1024 * 1024


def algorithmic_bytes(rows, cols, op, scale_kind="row"):
    n = rows * cols
    scale_bytes = 4 * rows if scale_kind == "row" else 4
    quant = 2 * n + n // 2 + n // 16 + scale_bytes
    if op == "quantize":
        return quant
    if op == "roundtrip":
        return quant + 2 * n
    if op == "dequantize":
        return n // 2 + n // 16 + scale_bytes + 2 * n
    if op == "residual":  # x in; codes, scales and row scale for x and for its residual out
        return 2 * n + 2 * (n // 2 + n // 16 + scale_bytes)
    if op == "guided":  # x, rollout amax, codes and scales in; codes out
        return 2 * n + n // 2 + n // 16 + scale_bytes + n // 2
    raise ValueError(op)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def fp4_tensor_peak():
    """Dense FP4 tensor peak: the measured BF16 GEMM burst figure times the nominal FP4/BF16 ratio
    (13.5 / 2.25 PFLOP/s dense = 6)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        return 6.0 * bf16, "measured bf16_tflops x 6 (nominal fp4/bf16)"
    except (OSError, KeyError, ValueError):
        return 6.0 * 1900.0, "fallback 1.9 PFLOP/s bf16 x 6 (nominal fp4/bf16)"


def recorded_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, if the kernels are unchanged."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_row_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    digest = h.hexdigest()[:16]
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and parts[0] == key and parts[2] == digest:
                    return float(parts[1])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value, world, device):
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def time_steps(fn, steps, warmup, world, device, graph=True):
    """W warm-up calls, then K timed calls bracketed by barrier + synchronize.  With `graph` the K
    calls are captured once into a CUDA graph and the timed region is one replay of it (host
    launch overhead out of the way, as in a captured training step); per-step times are then the
    replay time / K.  Returns (per-step device ms list, whole-region ms)."""
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(device)
    if graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.graph(g, stream=side):
            for _ in range(steps):
                fn()
        torch.cuda.synchronize(device)
        g.replay()  # one untimed replay
        torch.cuda.synchronize(device)
    barrier(world)
    torch.cuda.synchronize(device)
    if graph:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        g.replay()
        end.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        torch.cuda.synchronize(device)
        region = start.elapsed_time(end)
        return [region / steps] * steps, region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    torch.cuda.synchronize(device)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    region = starts[0].elapsed_time(ends[-1])
    return per, region


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_pass(x_u16, op, threads, scale_kind="row", mode="four_over_six"):
    """The oracle on the rows of x_u16, split into `threads` contiguous row ranges run at once
    (the ctypes calls release the GIL, so each range runs on its own core)."""
    import oracle

    omode = {"six": oracle.MODE_SIX, "four_over_six": oracle.MODE_FOUR_OVER_SIX,
             "four_over_six_fp16": oracle.MODE_FOUR_OVER_SIX_FP16}[mode]
    okind = oracle.SCALE_TENSOR if scale_kind == "tensor" else oracle.SCALE_ROW

    def one(part):
        out = oracle.quantize(part, omode, okind)
        if op != "quantize":
            oracle.dequantize(out["codes"], out["scales"], out["scale"], okind)

    if threads <= 1:
        one(x_u16)
        return
    from concurrent.futures import ThreadPoolExecutor

    bounds = [len(x_u16) * i // threads for i in range(threads + 1)]
    parts = [x_u16[bounds[i]:bounds[i + 1]] for i in range(threads) if bounds[i + 1] > bounds[i]]
    with ThreadPoolExecutor(max_workers=len(parts)) as pool:
        list(pool.map(one, parts))


def cpu_baseline(x, op, seconds, scale_kind="row", mode="four_over_six"):
    """The oracle, as it stands, on bounded samples of rows of x: once on one thread, once on all
    host cores (the reported value).  Each sample is sized for about seconds / 2 of CPU time."""
    import numpy as np

    from nvfp4_block_scaled_row_gb300 import synth

    rows, cols = x.shape
    probe = synth.as_u16(x[:2])
    t0 = time.perf_counter()
    oracle_pass(probe, op, 1, scale_kind, mode)
    per_row = (time.perf_counter() - t0) / 2
    cores = host_cores()
    res = {}
    for threads in (1, cores):
        n = int(max(4 * threads, min(rows, threads * seconds / 2 / max(per_row, 1e-6))))
        idx = np.linspace(0, rows - 1, n).astype(np.int64)
        sample = synth.as_u16(x[torch.as_tensor(idx, device=x.device)])
        t0 = time.perf_counter()
        oracle_pass(sample, op, threads, scale_kind, mode)
        dt = time.perf_counter() - t0
        res[threads] = (n, dt, algorithmic_bytes(n, cols, op, scale_kind) / dt / 1e9)
    what = "quantize+dequantize" if op != "quantize" else "quantize"
    n1, dt1, gbs1 = res[1]
    n, dt, gbs = res[cores]
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "elem_per_s": round(n * cols / dt, 1),
            "sample": f"{n} evenly spaced rows of the {rows}x{cols} workload, {what}, {dt:.1f} s "
                      f"on {cores} threads (one row range each)",
            "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                              "elem_per_s": round(n1 * cols / dt1, 1),
                              "sample": f"{n1} evenly spaced rows, {dt1:.1f} s"}}


def run_reference(args, world, rank):
    """--impl reference: the CPU oracle on the host cores, on the headline workload."""
    from nvfp4_block_scaled_row_gb300 import synth

    if rank != 0:
        return
    w = synth.workload(HEADLINE)
    # The steps sample rows of a 16384-row instance of the workload's recipe (same row
    # distribution: the zero and spike rows keep their fractions), so drawing it stays cheap.
    x = synth.generate(HEADLINE, device="cuda:0" if torch.cuda.is_available() else "cpu",
                       rows=min(w.rows, 16384))["x"]
    cores = host_cores()
    rows_per_step = 8 * cores
    total_rows = rows_per_step * (args.steps + args.warmup)
    idx = torch.linspace(0, x.shape[0] - 1, total_rows).long().to(x.device)
    xs = synth.as_u16(x[idx])
    times = []
    for s in range(args.warmup + args.steps):
        chunk = xs[s * rows_per_step:(s + 1) * rows_per_step]
        t0 = time.perf_counter()
        oracle_pass(chunk, "roundtrip", cores)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    step_bytes = algorithmic_bytes(rows_per_step, w.cols, "roundtrip")
    sec = statistics.mean(times)
    value = step_bytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name} (workload {w.index}) sample", "rows": w.rows,
                   "sampled_from_rows": x.shape[0],
                   "cols": w.cols, "rows_per_step": rows_per_step, "op": "roundtrip",
                   "scale": "row", "mode": "four_over_six"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} evenly spaced rows per step of a "
                                   f"{x.shape[0]}x{w.cols} draw of the {w.rows}-row recipe, "
                                   f"split over {cores} threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "elem_per_s": round(rows_per_step * w.cols / sec, 1),
    }
    print(json.dumps(line))


def bench_op(nv, x, op, kind, mode, steps, warmup, world, device, offsets=None):
    rows, cols = x.shape
    if op == "roundtrip":
        outs = nv.nvfp4_fused_roundtrip(x, kind, mode)
        codes, scales, scale, y = outs
        ws = torch.empty(nv.nvfp4_tensor_workspace_bytes(), dtype=torch.uint8, device=device)
        fn = lambda: nv.nvfp4_fused_roundtrip(x, kind, mode, codes, scales, scale, y, ws)
    elif op == "quantize" and kind == "row":
        codes, scales, scale = nv.nvfp4_quantize_rowwise(x, mode, offsets)
        fn = lambda: nv.nvfp4_quantize_rowwise(x, mode, offsets, codes, scales, scale)
    elif op == "quantize":
        codes, scales, scale = nv.nvfp4_quantize_tensor(x, mode)
        ws = torch.empty(nv.nvfp4_tensor_workspace_bytes(), dtype=torch.uint8, device=device)
        fn = lambda: nv.nvfp4_quantize_tensor(x, mode, codes, scales, scale, ws)
    elif op == "residual":
        fn = lambda: nv.nvfp4_quantize_residual(x, mode)
    elif op == "gemm":  # y = x . w^T, w = the first 2048 rows of the weight workload
        from nvfp4_block_scaled_row_gb300 import synth
        w = synth.generate(1, device=device)["x"][:, :cols].contiguous()
        xc, xs, xd = nv.nvfp4_quantize_rowwise(x, mode)
        wc, ws, wd = nv.nvfp4_quantize_tensor(w, mode)
        xsw, wsw = nv.nvfp4_swizzle_block_scales(xs, cols), nv.nvfp4_swizzle_block_scales(ws, cols)
        y = torch.empty((rows, w.shape[0]), dtype=torch.bfloat16, device=device)
        fn = lambda: nv.nvfp4_gemm_nt(xc, xsw, xd, wc, wsw, wd, y)
        per, region = time_steps(fn, steps, warmup, world, device)
        ms = statistics.mean(per)
        flops = 2.0 * rows * w.shape[0] * cols
        return {"gbs": flops / (ms * 1e-3) / 1e12, "ms": ms, "region_ms": region,
                "launches_per_step": 1, "unit": "TFLOP/s"}
    elif op == "guided":
        amax = nv.nvfp4_row_amax(x)
        rc, rs, _ = nv.nvfp4_quantize_rowwise(x, mode)
        out = torch.empty_like(rc)
        fn = lambda: nv.nvfp4_quantize_guided(x, amax, rc, rs, mode, out)
    else:  # dequantize
        codes, scales, scale = (nv.nvfp4_quantize_rowwise(x, mode) if kind == "row"
                                else nv.nvfp4_quantize_tensor(x, mode))
        y = torch.empty_like(x)
        fn = lambda: nv.nvfp4_dequantize(codes, scales, scale, kind, y)
    per, region = time_steps(fn, steps, warmup, world, device)
    ms = statistics.mean(per)
    gbs = algorithmic_bytes(rows, cols, op, kind) / (ms * 1e-3) / 1e9
    launches = 2 if (kind == "tensor" and op != "dequantize") else 1
    return {"gbs": gbs, "ms": ms, "region_ms": region, "launches_per_step": launches}


def e2e_roundtrip(nv, x, steps, warmup, device):
    """Public-API round trip of a host-resident matrix (nvfp4_fused_roundtrip_host): every step
    copies x host->device, runs the fused kernel and copies all outputs back (chunked and
    overlapped inside the call); timed on the host around a synchronize."""
    rows, cols = x.shape
    x_host = x.cpu().pin_memory()
    outs = nv.nvfp4_fused_roundtrip_host(x_host)
    ws = torch.empty(nv.nvfp4_roundtrip_host_workspace_bytes(cols), dtype=torch.uint8,
                     device=device)
    torch.cuda.synchronize(device)

    def step():
        nv.nvfp4_fused_roundtrip_host(x_host, "four_over_six", *outs, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize(device)
    sec = (time.perf_counter() - t0) / steps
    h2d = x.numel() * 2
    d2h = sum(t.numel() * t.element_size() for t in outs)
    gbs = algorithmic_bytes(rows, cols, "roundtrip") / sec / 1e9
    return {"value": round(gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(sec * 1e3, 3),
            "api": "nvfp4_fused_roundtrip_host (pinned host buffers, chunked, overlapped)"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads")
    ap.add_argument("--only", default=None, metavar="WORKLOAD/OP[/KIND[/MODE]]",
                    help="time one operation on one workload and print one short JSON line "
                         "(for profiling), e.g. moe_activation/roundtrip or "
                         "weight_expert_up/quantize/tensor/six")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        run_reference(args, world, rank)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import nvfp4_block_scaled_row_gb300 as nv
    from nvfp4_block_scaled_row_gb300 import synth

    nv.library()
    if args.only:
        parts = args.only.split("/")
        ww = synth.workload(parts[0] if not parts[0].isdigit() else int(parts[0]))
        op = parts[1]
        kind = parts[2] if len(parts) > 2 else ww.scale_kind
        mode = parts[3] if len(parts) > 3 else "four_over_six"
        d = synth.generate(ww.index, device=device)
        r = bench_op(nv, d["x"], op, kind, mode, args.steps, args.warmup, world, device,
                     d["offsets"] if op == "quantize" and kind == "row" else None)
        if rank == 0:
            print(json.dumps({"only": args.only, "shape": list(d["x"].shape),
                              "us_per_step": round(r["ms"] * 1e3, 2),
                              r.get("unit", "gbs"): round(r["gbs"], 1),
                              "device_status": nv.nvfp4_get_device_status()}))
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    w = synth.workload(HEADLINE)
    x = synth.generate(HEADLINE, device=device)["x"]
    rows, cols = x.shape

    # Headline: fused round trip on the largest workload, one replay of K captured launches timed
    # with events on the launching stream.
    with ClockSampler(local) as clocks:
        head = bench_op(nv, x, "roundtrip", "row", "four_over_six", args.steps, args.warmup,
                        world, device)
    ms = max_over_ranks(head["ms"], world, device)
    step_bytes = algorithmic_bytes(rows, cols, "roundtrip")
    value = world * step_bytes / (ms * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    achieved = step_bytes / (head["ms"] * 1e-3) / 1e9
    status = nv.nvfp4_get_device_status()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{w.name} (workload {w.index}): {w.summary}",
                   "rows": rows, "cols": cols, "op": "fused quantize->dequantize round trip",
                   "scale": "row (per-token)", "mode": "four_over_six",
                   "l2": f"inputs larger than L2 ({rows * cols * 2 / 1e6:.0f} MB > 129 MB), "
                         "no flush",
                   "timing": "K steps captured in one CUDA graph, one replay timed with CUDA "
                             "events",
                   "parallelism": f"replicas x{world}"},
        "elem_per_s": round(world * rows * cols / (ms * 1e-3), 1),
        "frac_of_hbm_peak": round(achieved / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic("fused_roundtrip_row_long_rollout"),
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one "
                                       "launch on this workload (profiles/dram_traffic.txt); "
                                       "null when the kernel sources changed since",
                     "kernel": "quantize_kernel<four_over_six, row, fused>",
                     "bytes_per_launch": step_bytes, "peak_source": f"{peak_src} hbm_gbs"},
        "gpu_launches": args.steps * head["launches_per_step"],
        "clocks": clocks.summary(),
        "device_status": status,
    }

    if rank == 0:
        line["e2e"] = e2e_roundtrip(nv, x, max(3, args.steps // 5), 3, device)
        line["cpu_baseline"] = cpu_baseline(x, "roundtrip", args.cpu_seconds)
    if not args.no_extras:
        also = {}
        del x
        torch.cuda.empty_cache()
        for idx, op, kind, mode in ((2, "roundtrip", "row", "four_over_six"),
                                    (3, "quantize", "row", "four_over_six"),
                                    (4, "quantize", "row", "four_over_six"),
                                    (4, "dequantize", "row", "four_over_six"),
                                    (1, "quantize", "tensor", "four_over_six"),
                                    (1, "quantize", "tensor", "six"),
                                    (1, "dequantize", "tensor", "four_over_six"),
                                    (0, "quantize", "row", "four_over_six"),
                                    (2, "quantize", "row", "four_over_six"),
                                    (2, "quantize", "row", "four_over_six_fp16"),
                                    (2, "residual", "row", "four_over_six"),
                                    (2, "guided", "row", "four_over_six"),
                                    (2, "gemm", "row", "four_over_six")):
            ww = synth.workload(idx)
            d = synth.generate(idx, device=device)
            r = bench_op(nv, d["x"], op, kind, mode, max(5, args.steps // 2), 3, world, device,
                         d["offsets"] if op == "quantize" and kind == "row" else None)
            if r.get("unit") == "TFLOP/s":
                fp4_peak, fp4_src = fp4_tensor_peak()
                also[f"{ww.name}/{op}/{kind}/{mode}"] = {
                    "tflops": round(r["gbs"], 1), "frac": round(r["gbs"] / fp4_peak, 4),
                    "peak_tflops": round(fp4_peak, 1), "peak_source": fp4_src,
                    "us_per_step": round(r["ms"] * 1e3, 2),
                    "shape": [d["x"].shape[0], 2048, d["x"].shape[1]]}
            else:
                also[f"{ww.name}/{op}/{kind}/{mode}"] = {
                    "gbs": round(r["gbs"], 1), "frac": round(r["gbs"] / peak, 4),
                    "us_per_launch": round(r["ms"] * 1e3, 2),
                    "elem_per_s": round(d["x"].numel() / (r["ms"] * 1e-3), 1),
                    "shape": list(d["x"].shape)}
            del d
            torch.cuda.empty_cache()
        line["also"] = also
        line["device_status_after_extras"] = nv.nvfp4_get_device_status()
        if rank == 0:
            # The oracle on a bounded sample of every workload, in the operation that workload
            # names (about cpu-seconds / 5 of CPU time each).
            cpus = {}
            for idx, op, kind, mode in ((0, "roundtrip", "row", "four_over_six"),
                                        (1, "roundtrip", "tensor", "four_over_six"),
                                        (2, "roundtrip", "row", "four_over_six"),
                                        (3, "quantize", "row", "four_over_six"),
                                        (4, "roundtrip", "row", "four_over_six")):
                ww = synth.workload(idx)
                d = synth.generate(idx, device=device)
                cb = cpu_baseline(d["x"], op, max(1.0, args.cpu_seconds / 5), kind, mode)
                cpus[f"{ww.name}/{op}/{kind}/{mode}"] = cb
                del d
                torch.cuda.empty_cache()
            line["cpu_baselines"] = cpus
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
