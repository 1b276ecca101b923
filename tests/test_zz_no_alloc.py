"""The allocation-free quantiser entry point, for callers that cannot allocate device memory
(for example a runtime that plans all device memory at start-up and allows no later allocation,
so it cannot hand nvfp4_quantize a workspace).  Its output must equal nvfp4_quantize's, bit for
bit, on two calls in a row: the second call uses a tensor with a much smaller amax, so a scratch
array that kept the first call's maxima would change its scales.

This file is named to be collected last, so a run that stops at the first failure has already
run every other test; it also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

from precision_moe_numerics_03_b300 import inputs, moe4

pytestmark = pytest.mark.gpu


def _reference(x, nmat, rows, cols, flags):
    codes = torch.empty((nmat, rows, cols // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((nmat, rows, cols // 16), dtype=torch.uint8, device="cuda")
    g = torch.empty(nmat, dtype=torch.float32, device="cuda")
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_NVFP4_QUANTIZE, nmat))
    moe4.nvfp4_quantize(x, nmat, rows, cols, cols, codes, sf, g, None, flags, ws)
    return codes, sf, g


def _noalloc(x, nmat, rows, cols, flags):
    codes = torch.empty((nmat, rows, cols // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((nmat, rows, cols // 16), dtype=torch.uint8, device="cuda")
    g = torch.empty(nmat, dtype=torch.float32, device="cuda")
    moe4.nvfp4_quantize_noalloc(x, nmat, rows, cols, cols, codes, sf, g, flags)
    return codes, sf, g


def test_noalloc_matches_workspace_entry_point_twice():
    moe4.load()
    rng = np.random.default_rng(77)
    cases = [
        (3, 256, 512, 1000.0, moe4.FOUR_OVER_SIX),                      # large values first
        (3, 256, 512, 0.001, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT),  # then much smaller ones
    ]
    for nmat, rows, cols, scale, flags in cases:
        x = inputs.to_bf16_bits((rng.standard_t(3, (nmat * rows, cols)) * scale).astype(np.float32))
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        want = _reference(xd, nmat, rows, cols, flags)
        got = _noalloc(xd, nmat, rows, cols, flags)
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a, b)


def test_noalloc_rejects_too_many_matrices():
    lib = moe4.load()
    assert lib.nvfp4_quantize_noalloc(1 << 20, 4097, 16, 16, 16, 1 << 20, 1 << 20, 1 << 20, 1, None) == moe4.ERR_ARG
