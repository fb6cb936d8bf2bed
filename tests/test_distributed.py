"""Multi-rank host logic on CPU gloo ranks: row sharding needs no exchange, and the sharded
per-tensor path (shard amax -> max over ranks -> encode with that amax) is bit-identical to the
unsharded result.  The per-rank compute here is the CPU oracle."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from nvfp4_block_scaled_row_gb300 import distributed as D
from nvfp4_block_scaled_row_gb300 import synth

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, xb, offsets, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        rows = xb.shape[0]
        # Per-tensor: local amax, max over ranks, encode the shard with the global amax.
        a, b = D.shard_rows(rows, WORLD, rank)
        shard = np.ascontiguousarray(xb[a:b])
        local = torch.tensor([oracle.amax(shard)], dtype=torch.float32)
        D.global_amax(local)
        t = oracle.quantize_given_amax(shard, float(local.item()))
        # Per-token over expert groups: no exchange at all.
        ga, gb = D.shard_groups(offsets, WORLD, rank)
        r = oracle.quantize(np.ascontiguousarray(xb[ga:gb]))
        results[rank] = {"tensor": t, "amax": float(local.item()), "rows": (a, b),
                         "groups": (ga, gb), "row": r}
    finally:
        dist.destroy_process_group()


def test_sharded_tensor_and_row_paths_match_unsharded():
    d = synth.generate(3, rows=320)
    xb = synth.as_u16(d["x"])
    offsets = d["offsets"]
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(port, xb, offsets, results), nprocs=WORLD,
                           start_method="spawn", join=True)
        res = dict(results)
    whole = oracle.quantize(xb, scale_kind=oracle.SCALE_TENSOR)
    assert {r["amax"] for r in res.values()} == {oracle.amax(xb)}
    codes = np.concatenate([res[r]["tensor"]["codes"] for r in range(WORLD)])
    scales = np.concatenate([res[r]["tensor"]["scales"] for r in range(WORLD)])
    assert np.array_equal(codes, whole["codes"]) and np.array_equal(scales, whole["scales"])
    for r in range(WORLD):
        assert res[r]["tensor"]["scale"].view(np.uint32)[0] == whole["scale"].view(np.uint32)[0]
    per_token = oracle.quantize(xb)
    assert res[0]["groups"][0] == 0 and res[WORLD - 1]["groups"][1] == xb.shape[0]
    assert res[0]["groups"][1] == res[1]["groups"][0]
    got = np.concatenate([res[r]["row"]["codes"] for r in range(WORLD)])
    assert np.array_equal(got, per_token["codes"])


def test_shard_rows_cover_exactly():
    for rows in (0, 1, 5, 16384, 32853):
        for world in (1, 2, 3, 8):
            spans = [D.shard_rows(rows, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_shard_groups_align_to_group_boundaries():
    off = synth.generate(3, rows=2560)["offsets"]
    offs = off.tolist()
    for world in (1, 2, 4):
        spans = [D.shard_groups(off, world, r) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == offs[-1]
        for a, b in spans:
            assert a in offs and b in offs and a <= b
        assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
