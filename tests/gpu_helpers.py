"""Helpers for the GPU parity tests: move seeded host inputs to the device, call the library
through its C ABI (the ctypes binding), and bring results back for comparison with the oracle."""
import numpy as np
import torch

from precision_moe_numerics_03_b300 import moe4

DEV = "cuda"


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(DEV)
    return torch.from_numpy(a).to(DEV)


def to_np(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def empty_u8(*shape):
    return torch.empty(shape, dtype=torch.uint8, device=DEV)


def nvfp4_quantize(x_bits: torch.Tensor, nmat, rows, cols, flags=moe4.FOUR_OVER_SIX, amax=None, ld=None):
    """x_bits: device int16 tensor holding bf16 bits, [nmat*rows, ld]."""
    ld = cols if ld is None else ld
    codes = empty_u8(nmat, rows, cols // 2)
    sf = empty_u8(nmat, rows, cols // 16)
    g = torch.empty(nmat, dtype=torch.float32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_NVFP4_QUANTIZE, nmat))
    amax_t = None
    if amax is not None:
        amax_t = torch.tensor(np.asarray(amax, np.float32).reshape(-1), device=DEV)
        flags |= moe4.AMAX_GIVEN
    moe4.nvfp4_quantize(x_bits, nmat, rows, cols, ld, codes, sf, g, amax_t, flags, ws)
    torch.cuda.synchronize()
    return codes, sf, g


def first_mismatch(a: np.ndarray, b: np.ndarray):
    bad = np.argwhere(a != b)
    if bad.size == 0:
        return None
    i = tuple(bad[0])
    return "first mismatch at %s: got %r want %r (%d mismatches of %d)" % (i, a[i], b[i], len(bad), a.size)


def mma_layout(e8: torch.Tensor, rows: int, nblk: int) -> torch.Tensor:
    """Canonical scale bytes [rows, nblk] rearranged by the library's own layout change."""
    out = torch.empty(rows * nblk, dtype=torch.uint8, device=e8.device)
    moe4.moe4_sf_to_mma_layout(e8, 1, rows, nblk, out)
    return out
