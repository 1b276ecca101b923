"""Thin ctypes binding of libmoe4.so (include/moe4.h): the same entry-point names, torch tensors
in place of device pointers, the current torch CUDA stream unless one is given.

This module only marshals arguments.  Every step of the computation runs in the library's CUDA
kernels; there is no Python or CPU fallback, and `load()` raises when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe4.so")

OK, ERR_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = 0, -1, -2, -3, -4, -5
FOUR_OVER_SIX = 0x00001
AMAX_GIVEN = 0x00002
SR = 0x00004
ROWWISE = 0x00010
COLWISE = 0x00020
OUT_F32 = 0x00100
OUT_BF16 = 0x00200
GROUP_M = 0x01000
GROUP_K = 0x02000
ACCUMULATE = 0x04000
SF_MMA_LAYOUT = 0x10000
MXFP8 = 0x20000
SF_OUT_MMA = 0x40000
PASS_QUANT = 0x100000
PASS_REQUANT = 0x200000
SHARE_SMS = 0x400000

OP_NVFP4_QUANTIZE = 1
OP_HADAMARD_QUANT = 2
OP_PERMUTE_PLAN = 3

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_u32 = ctypes.c_uint32
_int = ctypes.c_int
_sz = ctypes.c_size_t
_f32 = ctypes.c_float

_SIGNATURES = {
    "moe4_version": (_int, []),
    "moe4_status_string": (ctypes.c_char_p, [_int]),
    "moe4_workspace_size": (_sz, [_int, _i64, _i64, _i64]),
    "moe4_workspace_size_gemm": (_sz, [_int, _i64, _i64, _i64, _i64]),
    "moe4_get_status": (_int, [_vp]),
    "moe4_selftest_wait": (_int, [_i64, _vp]),
    "moe4_tensor_peak_probe": (_int, [_int, _i64, _i64, _vp, _vp]),
    "moe4_check_group_offsets": (_int, [_vp, _i64, _i64, _i64]),
    "nvfp4_quantize": (_int, [_vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _u32, _vp, _sz, _vp]),
    "nvfp4_quantize_f32": (_int, [_vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _u32, _vp, _sz, _vp]),
    "nvfp4_quantize_noalloc": (_int, [_vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _u32, _vp]),
    "nvfp4_dequantize": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _u32, _vp]),
    "mxfp8_requant_transpose_sr": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _u64, _u32, _u32, _vp]),
    "nvfp4_quantize_f32_requant": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _u64, _u32, _i64,
                                          _vp, _u32, _vp]),
    "mxfp8_quantize": (_int, [_vp, _i64, _i64, _vp, _vp, _u64, _u32, _u32, _vp]),
    "mxfp8_quantize_rowcol": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _u32, _vp]),
    "hadamard_quant": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _u32, _vp, _sz, _vp]),
    "hadamard_dequant": (_int, [_vp, _vp, _vp, _i64, _i64, _vp, _u32, _vp]),
    "grouped_expert_gemm_nvfp4": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _u32,
                                         _vp, _sz, _vp]),
    "grouped_expert_gemm_nvfp4_hadamard_amax": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                                        _vp, _vp, _u32, _vp, _sz, _vp]),
    "grouped_expert_gemm_nvfp4_swiglu": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                                _vp, _vp, _vp, _u32, _vp, _sz, _vp]),
    "grouped_expert_gemm_nvfp4_hadamard_mx": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                                      _vp, _vp, _u32, _vp, _sz, _vp]),
    "grouped_gemm_mxfp8": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _u32, _vp, _sz, _vp]),
    "grouped_gemm_mxfp8_swiglu_backward": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _u32,
                                                  _vp, _sz, _vp]),
    "grouped_gemm_mxfp8_wgrad_sgd": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _f32, _vp,
                                            _u32, _vp, _sz, _vp]),
    "moe4_sf_to_mma_layout": (_int, [_vp, _i64, _i64, _i64, _vp, _vp]),
    "moe4_route_topk": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "moe4_permute_plan": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _i64, _vp, _sz, _vp]),
    "moe4_permute_nvfp4": (_int, [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _u32, _vp]),
    "moe4_swiglu_backward": (_int, [_vp, _vp, _i64, _i64, _vp, _vp]),
    "moe4_swiglu_backward_mxfp8": (_int, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _u32, _vp]),
    "moe4_combine_backward": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "moe4_combine_backward_mxfp8": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _u32,
                                           _vp]),
    "moe4_swiglu": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "moe4_swiglu_amax": (_int, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "moe4_combine": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    "moe4_combine_hadamard": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    "moe4_dispatch_backward": (_int, [_vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    "moe4_sgd_update": (_int, [_vp, _vp, _i64, _f32, _vp, _vp]),
    "moe4_convert": (_int, [_int, _vp, _i64, _vp, _vp]),
    "moe4_sr_words": (_int, [_u64, _u32, _u64, _i64, _vp, _vp]),
}

_LIB = None


class Moe4Error(RuntimeError):
    def __init__(self, name: str, status: int):
        msg = load().moe4_status_string(status).decode()
        super().__init__("%s failed: %s (status %d)" % (name, msg, status))
        self.status = status


def load() -> ctypes.CDLL:
    """Open libmoe4.so.  Raises if it has not been built: there is no fallback path."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe4.so is missing (%s); build it with "
                               "`python -m precision_moe_numerics_03_b300.build`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def exported_symbols():
    return list(_SIGNATURES)


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe4 takes device tensors only")
    if not t.is_contiguous():
        raise ValueError("libmoe4 takes contiguous tensors only")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _ws_bytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def _call(name, *args):
    rc = getattr(load(), name)(*args)
    if rc != OK:
        raise Moe4Error(name, rc)


# ------------------------------------------------------------------ library
def moe4_version() -> int:
    return load().moe4_version()


def moe4_workspace_size(op: int, a: int = 0, b: int = 0, c: int = 0) -> int:
    return load().moe4_workspace_size(op, a, b, c)


def moe4_workspace_size_gemm(kind: int, a_rows: int, E: int, b_rows: int, K: int) -> int:
    return load().moe4_workspace_size_gemm(kind, a_rows, E, b_rows, K)


def moe4_get_status(stream=None) -> int:
    return load().moe4_get_status(_s(stream))


def moe4_check_group_offsets(offs, total: int, align: int = 128):
    """Host-side check of group offsets (a host array or CPU tensor of E+1 int32 values)."""
    import numpy as np
    a = np.ascontiguousarray(offs.cpu().numpy() if hasattr(offs, "cpu") else offs, dtype=np.int32)
    _call("moe4_check_group_offsets", a.ctypes.data, a.size - 1, total, align)


def moe4_selftest_wait(limit_cycles, stream=None):
    _call("moe4_selftest_wait", limit_cycles, _s(stream))


def moe4_tensor_peak_probe(kind, iters, ctas, sink, stream=None):
    _call("moe4_tensor_peak_probe", kind, iters, ctas, _p(sink), _s(stream))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned scratch buffer of at least nbytes (torch's allocator aligns to 512)."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ NVFP4 / MXFP8 / Hadamard
def nvfp4_quantize(x, nmat, rows, cols, ld, codes, sf, g_dec, amax_in=None, flags=FOUR_OVER_SIX, ws=None,
                   stream=None):
    _call("nvfp4_quantize", _p(x), nmat, rows, cols, ld, _p(codes), _p(sf), _p(g_dec), _p(amax_in), flags,
          _p(ws), _ws_bytes(ws), _s(stream))


def nvfp4_quantize_f32(x, nmat, rows, cols, ld, codes, sf, g_dec, amax_in=None, flags=FOUR_OVER_SIX, ws=None,
                       stream=None):
    _call("nvfp4_quantize_f32", _p(x), nmat, rows, cols, ld, _p(codes), _p(sf), _p(g_dec), _p(amax_in), flags,
          _p(ws), _ws_bytes(ws), _s(stream))


def nvfp4_quantize_noalloc(x, nmat, rows, cols, ld, codes, sf, g_dec, flags=FOUR_OVER_SIX, stream=None):
    """nvfp4_quantize without a caller-provided workspace: its scratch is a fixed array owned by
    the library (at most 4096 matrices per call; overlapping calls race on it)."""
    _call("nvfp4_quantize_noalloc", _p(x), nmat, rows, cols, ld, _p(codes), _p(sf), _p(g_dec), flags, _s(stream))


def nvfp4_dequantize(codes, sf, g_dec, nmat, rows, cols, out, flags=OUT_BF16, stream=None):
    _call("nvfp4_dequantize", _p(codes), _p(sf), _p(g_dec), nmat, rows, cols, _p(out), flags, _s(stream))


def mxfp8_requant_transpose_sr(codes, sf, g_dec, nmat, rows, cols, q_t, e8_t, seed=0, stream_id=0, flags=SR,
                               stream=None):
    _call("mxfp8_requant_transpose_sr", _p(codes), _p(sf), _p(g_dec), nmat, rows, cols, _p(q_t), _p(e8_t),
          seed, stream_id, flags, _s(stream))


def nvfp4_quantize_f32_requant(x, nmat, rows, cols, amax_in, codes, sf, g_dec, q_t, e8_t, seed=0, stream_id=0,
                               group_offs=None, flags=FOUR_OVER_SIX | SR, stream=None, mat_base=0):
    _call("nvfp4_quantize_f32_requant", _p(x), nmat, rows, cols, _p(amax_in), _p(codes), _p(sf), _p(g_dec), _p(q_t),
          _p(e8_t), seed, stream_id, mat_base, _p(group_offs), flags, _s(stream))


def mxfp8_quantize(x, rows, cols, q, e8, seed=0, stream_id=0, flags=ROWWISE, stream=None):
    _call("mxfp8_quantize", _p(x), rows, cols, _p(q), _p(e8), seed, stream_id, flags, _s(stream))


def mxfp8_quantize_rowcol(x, rows, cols, q_row, e8_row, q_col, e8_col, flags=0, stream=None):
    _call("mxfp8_quantize_rowcol", _p(x), rows, cols, _p(q_row), _p(e8_row), _p(q_col), _p(e8_col), flags,
          _s(stream))


def hadamard_quant(x, rows, cols, codes, sf, g_dec, flags=FOUR_OVER_SIX, ws=None, stream=None):
    _call("hadamard_quant", _p(x), rows, cols, _p(codes), _p(sf), _p(g_dec), flags, _p(ws), _ws_bytes(ws),
          _s(stream))


def hadamard_dequant(codes, sf, g_dec, rows, cols, out, flags=0, stream=None):
    _call("hadamard_dequant", _p(codes), _p(sf), _p(g_dec), rows, cols, _p(out), flags, _s(stream))


# ------------------------------------------------------------------ GEMMs
def grouped_expert_gemm_nvfp4(a_codes, a_sf, a_g_dec, b_codes, b_sf, b_g_dec, group_offs, E, rows_total, N, K, d,
                              flags=OUT_F32, ws=None, stream=None):
    _call("grouped_expert_gemm_nvfp4", _p(a_codes), _p(a_sf), _p(a_g_dec), _p(b_codes), _p(b_sf), _p(b_g_dec),
          _p(group_offs), E, rows_total, N, K, _p(d), flags, _p(ws), _ws_bytes(ws), _s(stream))


def grouped_expert_gemm_nvfp4_hadamard_amax(a_codes, a_sf, a_g_dec, b_codes, b_sf, b_g_dec, group_offs, E,
                                            rows_total, N, K, d, amax_out, flags=0, ws=None, stream=None):
    _call("grouped_expert_gemm_nvfp4_hadamard_amax", _p(a_codes), _p(a_sf), _p(a_g_dec), _p(b_codes), _p(b_sf),
          _p(b_g_dec), _p(group_offs), E, rows_total, N, K, _p(d), _p(amax_out), flags, _p(ws), _ws_bytes(ws),
          _s(stream))


def grouped_expert_gemm_nvfp4_swiglu(a_codes, a_sf, a_g_dec, b_codes, b_sf, b_g_dec, group_offs, E, rows_total, f, K,
                                     gu, h, amax_out, flags=0, ws=None, stream=None):
    _call("grouped_expert_gemm_nvfp4_swiglu", _p(a_codes), _p(a_sf), _p(a_g_dec), _p(b_codes), _p(b_sf),
          _p(b_g_dec), _p(group_offs), E, rows_total, f, K, _p(gu), _p(h), _p(amax_out), flags, _p(ws), _ws_bytes(ws),
          _s(stream))


def grouped_expert_gemm_nvfp4_hadamard_mx(a_codes, a_sf, a_g_dec, b_codes, b_sf, b_g_dec, group_offs, E, rows_total,
                                          N, K, q, e8, flags=0, ws=None, stream=None):
    _call("grouped_expert_gemm_nvfp4_hadamard_mx", _p(a_codes), _p(a_sf), _p(a_g_dec), _p(b_codes), _p(b_sf),
          _p(b_g_dec), _p(group_offs), E, rows_total, N, K, _p(q), _p(e8), flags, _p(ws), _ws_bytes(ws), _s(stream))


def grouped_gemm_mxfp8(a, a_e8, b, b_e8, group_offs, E, M, N, K, d, flags=OUT_F32 | GROUP_M, ws=None,
                       stream=None):
    _call("grouped_gemm_mxfp8", _p(a), _p(a_e8), _p(b), _p(b_e8), _p(group_offs), E, M, N, K, _p(d), flags,
          _p(ws), _ws_bytes(ws), _s(stream))


def grouped_gemm_mxfp8_swiglu_backward(a, a_e8, b, b_e8, group_offs, E, M, f, K, gu, dgu, flags=0, ws=None,
                                       stream=None):
    _call("grouped_gemm_mxfp8_swiglu_backward", _p(a), _p(a_e8), _p(b), _p(b_e8), _p(group_offs), E, M, f, K, _p(gu),
          _p(dgu), flags, _p(ws), _ws_bytes(ws), _s(stream))


def grouped_gemm_mxfp8_wgrad_sgd(a, a_e8, b, b_e8, group_offs, E, M, N, K, w32, w_bf16, lr, amax_out, flags=0,
                                 ws=None, stream=None):
    _call("grouped_gemm_mxfp8_wgrad_sgd", _p(a), _p(a_e8), _p(b), _p(b_e8), _p(group_offs), E, M, N, K, _p(w32),
          _p(w_bf16), float(lr), _p(amax_out), flags, _p(ws), _ws_bytes(ws), _s(stream))


def moe4_sf_to_mma_layout(sf, nmat, rows, nblk, out, stream=None):
    _call("moe4_sf_to_mma_layout", _p(sf), nmat, rows, nblk, _p(out), _s(stream))


# ------------------------------------------------------------------ routing and dispatch
def moe4_route_topk(logits, T, E, k, idx, w, stream=None):
    _call("moe4_route_topk", _p(logits), T, E, k, _p(idx), _p(w), _s(stream))


def moe4_permute_plan(idx, T, k, E, offs, row_of, src_of, rows_cap, ws, stream=None):
    _call("moe4_permute_plan", _p(idx), T, k, E, _p(offs), _p(row_of), _p(src_of), rows_cap, _p(ws),
          _ws_bytes(ws), _s(stream))


def moe4_permute_nvfp4(codes, sf, T, cols, src_of, rows_total, out_codes, out_sf, flags=0, stream=None):
    _call("moe4_permute_nvfp4", _p(codes), _p(sf), T, cols, _p(src_of), rows_total, _p(out_codes), _p(out_sf),
          flags, _s(stream))


def moe4_swiglu_backward(gu, dh, rows, f, dgu, stream=None):
    _call("moe4_swiglu_backward", _p(gu), _p(dh), rows, f, _p(dgu), _s(stream))


def moe4_swiglu_backward_mxfp8(gu, dh, rows, f, q_row, e8_row, q_col, e8_col, flags=0, stream=None):
    _call("moe4_swiglu_backward_mxfp8", _p(gu), _p(dh), rows, f, _p(q_row), _p(e8_row), _p(q_col), _p(e8_col), flags,
          _s(stream))


def moe4_combine_backward(dy, row_of, w, src_of, T, k, d, rows_total, dyhat, stream=None):
    _call("moe4_combine_backward", _p(dy), _p(row_of), _p(w), _p(src_of), T, k, d, rows_total, _p(dyhat),
          _s(stream))


def moe4_swiglu(gu, rows, f, h, stream=None):
    _call("moe4_swiglu", _p(gu), rows, f, _p(h), _s(stream))


def moe4_swiglu_amax(gu, rows, f, h, amax_out, stream=None):
    _call("moe4_swiglu_amax", _p(gu), rows, f, _p(h), _p(amax_out), _s(stream))


def moe4_combine_backward_mxfp8(dy, row_of, w, src_of, T, k, d, rows_total, q_row, e8_row, q_col, e8_col, flags=0,
                                stream=None):
    _call("moe4_combine_backward_mxfp8", _p(dy), _p(row_of), _p(w), _p(src_of), T, k, d, rows_total, _p(q_row),
          _p(e8_row), _p(q_col), _p(e8_col), flags, _s(stream))


def moe4_combine(yhat, row_of, w, T, k, d, y, stream=None):
    _call("moe4_combine", _p(yhat), _p(row_of), _p(w), T, k, d, _p(y), _s(stream))


def moe4_combine_hadamard(codes, sf, g_dec, row_of, w, T, k, d, y, stream=None):
    _call("moe4_combine_hadamard", _p(codes), _p(sf), _p(g_dec), _p(row_of), _p(w), T, k, d, _p(y), _s(stream))


def moe4_dispatch_backward(dxp, row_of, T, k, d, dx, stream=None):
    _call("moe4_dispatch_backward", _p(dxp), _p(row_of), T, k, d, _p(dx), _s(stream))


def moe4_sgd_update(w32, dw, n, lr, w_bf16, stream=None):
    _call("moe4_sgd_update", _p(w32), _p(dw), n, float(lr), _p(w_bf16), _s(stream))


# ------------------------------------------------------------------ checks of the device conversions
def moe4_convert(kind, x, n, out, stream=None):
    _call("moe4_convert", kind, _p(x), n, _p(out), _s(stream))


def moe4_sr_words(seed, stream_id, idx_base, n, out, stream=None):
    _call("moe4_sr_words", seed, stream_id, idx_base, n, _p(out), _s(stream))
