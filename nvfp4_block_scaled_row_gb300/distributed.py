"""Multi-GPU use of the quantizer: row sharding and the per-tensor amax exchange.

Per-token quantization ("NVFP4 RL" blog, Sec. 2) makes every row independent, so rows (or whole
expert groups) are split across ranks with no collective at all.  Per-tensor quantization of a
weight sharded across ranks ("NVFP4 RL" blog, Sec. 4, 4/6 for weights) has exactly one exchange:
the max over ranks of each shard's FP32 amax.  Max is exact and order-free, so the sharded result
is bit-identical to quantizing the whole tensor on one device.

The functions take an optional process group and work with any torch.distributed backend (NCCL
for CUDA tensors, gloo for CPU tensors).
"""
import torch
import torch.distributed as dist


def _world(group):
    if not dist.is_available() or not dist.is_initialized():
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def shard_rows(rows, world_size, rank):
    """Contiguous, near-equal row range [start, stop) of `rank` out of `world_size`."""
    if world_size < 1 or not 0 <= rank < world_size or rows < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(rows, world_size)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_groups(offsets, world_size, rank):
    """Row range [start, stop) covering whole expert groups, with the groups split into
    contiguous runs of near-equal row counts.  `offsets` is the int32 [G+1] group-offset list."""
    offs = [int(v) for v in torch.as_tensor(offsets).cpu().tolist()]
    total = offs[-1]
    g = len(offs) - 1

    def boundary(r):
        if r == 0:
            return 0
        if r == world_size:
            return g
        target = total * r / world_size
        best = min(range(g + 1), key=lambda i: (abs(offs[i] - target), i))
        return best

    lo, hi = boundary(rank), boundary(rank + 1)
    hi = max(hi, lo)
    return offs[lo], offs[hi]


def global_amax(local_amax, group=None):
    """In-place max over ranks of a float32 [1] tensor (the shard amax); returns it."""
    world, _ = _world(group)
    if world > 1:
        dist.all_reduce(local_amax, op=dist.ReduceOp.MAX, group=group)
    return local_amax


def quantize_tensor_sharded(x_local, mode="four_over_six", group=None, stream=None):
    """Per-tensor quantization of this rank's shard with the amax of the whole (sharded)
    tensor: local amax on the GPU, max over ranks, then the encoder with that amax."""
    from . import nvfp4_quantize_tensor_with_amax, nvfp4_tensor_amax

    amax = nvfp4_tensor_amax(x_local, stream=stream)
    global_amax(amax, group)
    return nvfp4_quantize_tensor_with_amax(x_local, amax, mode, stream=stream)
