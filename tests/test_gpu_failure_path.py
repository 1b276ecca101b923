"""The failure path of the bounded waits, without a GPU fault: a wait that nothing completes
gives up after its limit, moe4_get_status reports MOE4_ERR_TIMEOUT once, and the context keeps
working (a quantisation and a GEMM after it are still bit-exact / correct)."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import inputs, moe4
from gpu_helpers import DEV, first_mismatch, nvfp4_quantize, to_dev, to_np

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    moe4.load()
    assert moe4.moe4_get_status() == moe4.OK
    moe4.moe4_selftest_wait(1 << 24)  # ~8 ms of SM clock
    assert moe4.moe4_get_status() == moe4.ERR_TIMEOUT
    assert moe4.moe4_get_status() == moe4.OK  # read and cleared
    x = inputs.to_bf16_bits(np.random.default_rng(3).standard_normal((64, 256)).astype(np.float32))
    c, s, g = nvfp4_quantize(to_dev(x), 1, 64, 256)
    rc, rs, rg = oracle.nvfp4_quantize(oracle.bf16_to_f32(x))
    assert first_mismatch(to_np(c)[0], rc) is None and first_mismatch(to_np(s)[0], rs) is None
    assert moe4.moe4_get_status() == moe4.OK


def test_selftest_rejects_bad_limits():
    moe4.load()
    for bad in (0, (1 << 32) + 1):
        with pytest.raises(RuntimeError):
            moe4.moe4_selftest_wait(bad)
