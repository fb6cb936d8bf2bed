"""The allocation-free per-tensor entry point, called through the C ABI.

nvfp4_quantize_tensor_noalloc serves callers that cannot allocate device memory (allocator
callbacks, plugins handed only their tensors): its scratch is a fixed device array inside the
library instead of a caller workspace.  Its results must equal nvfp4_quantize_tensor's bit for
bit, on consecutive calls (the array keeps the previous call's contents) and on inputs with a
different amax.  This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import pytest
import torch

import nvfp4_block_scaled_row_gb300 as nv
from nvfp4_block_scaled_row_gb300 import build as nvbuild
from nvfp4_block_scaled_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return nv.library()


def _noalloc(lib, x, mode):
    rows, cols = x.shape
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=DEV)
    scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=DEV)
    ts = torch.empty(1, dtype=torch.float32, device=DEV)
    st = lib.nvfp4_quantize_tensor_noalloc(
        ctypes.c_void_p(x.data_ptr()), rows, cols, mode, ctypes.c_void_p(codes.data_ptr()),
        ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(ts.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, nv.nvfp4_status_string(st)
    torch.cuda.synchronize()
    return codes, scales, ts


@pytest.mark.parametrize("mode", [1, 0, 2])
def test_noalloc_matches_workspace_entry_point(lib, mode):
    name = {0: "six", 1: "four_over_six", 2: "four_over_six_fp16"}[mode]
    # The last input is one 4x2048 tensor: its amax pass writes fewer partial maxima than the
    # calls before it left in the shared array, so a read past them would change its result.
    inputs = [synth.generate(1, device=DEV)["x"],                 # weights, amax ~0.4
              synth.generate(4, device=DEV, rows=1024)["x"],       # spikes, amax 3e4
              synth.generate(0, device=DEV, rows=4)["x"]]          # tiny: one partial maximum
    for x in inputs:
        want = nv.nvfp4_quantize_tensor(x, name)
        torch.cuda.synchronize()
        for _ in range(2):  # two calls in a row through the shared array
            got = _noalloc(lib, x, mode)
            for a, b in zip(want, got):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert nv.nvfp4_get_device_status() == 0


def test_noalloc_rejects_bad_arguments_before_launch(lib):
    x = synth.generate(0, device=DEV, rows=4)["x"]
    P = ctypes.c_void_p
    assert lib.nvfp4_quantize_tensor_noalloc(P(x.data_ptr()), 4, 24, 1, P(0), P(0), P(0),
                                             None) == 2
    assert lib.nvfp4_quantize_tensor_noalloc(P(x.data_ptr()), 0, 2048, 1, None, None, None,
                                             None) == 0
