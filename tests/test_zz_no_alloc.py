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


_RESET_CHILD = r"""
import ctypes, sys
import numpy as np
lib = ctypes.CDLL(sys.argv[1])
vp, i64, u32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
lib.cudaMalloc.argtypes = [ctypes.POINTER(vp), sz]
lib.cudaMemcpy.argtypes = [vp, vp, sz, ctypes.c_int]
lib.cudaFree.argtypes = [vp]
lib.nvfp4_quantize_noalloc.argtypes = [vp, i64, i64, i64, i64, vp, vp, vp, u32, vp]
lib.nvfp4_quantize.argtypes = [vp, i64, i64, i64, i64, vp, vp, vp, vp, u32, vp, sz, vp]
H2D, D2H = 1, 2
nmat, rows, cols, flags = 3, 256, 512, 1  # Four Over Six


def must(rc, what):
    if rc != 0:
        raise SystemExit("%s returned %d" % (what, rc))


def quantize(x, noalloc):
    bufs = {}
    for name, n in (("x", x.nbytes), ("codes", nmat * rows * cols // 2), ("sf", nmat * rows * cols // 16),
                    ("g", 4 * nmat), ("ws", 4 * nmat)):
        p = vp()
        must(lib.cudaMalloc(ctypes.byref(p), n), "cudaMalloc")
        bufs[name] = p
    must(lib.cudaMemcpy(bufs["x"], x.ctypes.data, x.nbytes, H2D), "cudaMemcpy")
    if noalloc:
        must(lib.nvfp4_quantize_noalloc(bufs["x"], nmat, rows, cols, cols, bufs["codes"], bufs["sf"], bufs["g"],
                                        flags, None), "nvfp4_quantize_noalloc")
    else:
        must(lib.nvfp4_quantize(bufs["x"], nmat, rows, cols, cols, bufs["codes"], bufs["sf"], bufs["g"], None,
                                flags, bufs["ws"], 4 * nmat, None), "nvfp4_quantize")
    must(lib.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
    out = [np.empty(nmat * rows * cols // 2, np.uint8), np.empty(nmat * rows * cols // 16, np.uint8),
           np.empty(nmat, np.float32)]
    for a, name in zip(out, ("codes", "sf", "g")):
        must(lib.cudaMemcpy(a.ctypes.data, bufs[name], a.nbytes, D2H), "cudaMemcpy")
    for p in bufs.values():
        must(lib.cudaFree(p), "cudaFree")
    return out


def bf16_bits(v):
    u = v.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


rng = np.random.default_rng(78)
big = bf16_bits(rng.standard_t(3, (nmat * rows, cols)) * 1000.0)
small = bf16_bits(rng.standard_t(3, (nmat * rows, cols)) * 0.001)
must(lib.cudaSetDevice(0), "cudaSetDevice")
want_big = quantize(big, False)
got_big = quantize(big, True)
must(lib.cudaDeviceReset(), "cudaDeviceReset")  # a new context: the library's device data moves
got_small = quantize(small, True)
want_small = quantize(small, False)
got_small2 = quantize(small, True)
for got, want in ((got_big, want_big), (got_small, want_small), (got_small2, want_small)):
    for a, b in zip(got, want):
        if not np.array_equal(a, b):
            raise SystemExit("allocation-free output differs from nvfp4_quantize")
print("ok")
"""


def test_noalloc_after_device_reset():
    """A caller that tears its context down (cudaDeviceReset) and goes on: the allocation-free call
    must find its scratch array in the new context.  Runs in a child process that manages device
    memory with the CUDA runtime only (no torch), so resetting the device there leaves this
    process's context alone."""
    import subprocess
    import sys
    out = subprocess.run([sys.executable, "-c", _RESET_CHILD, moe4.LIB_PATH], capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
