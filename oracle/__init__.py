"""The oracle: a plain, slow CPU definition of the 4-bit MoE expert-layer numerics.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library (``precision_moe_numerics_03_b300``) and never imports it.

The element-wise and block-wise arithmetic lives in ``moe4_oracle.c`` (binary32 operations in the
written order, no fused multiply-add).  This module loads it with ctypes and adds the steps that
are plain array bookkeeping or need a library primitive: routing, permutation, SwiGLU, combine,
the SGD update and the float64 reference GEMMs.

Pages cited (the method is described in prose only):
  [DEBUT]  "Inkling 2 Small's Native 4-Bit Training: Debut and Doubts", "Confirmed" list.
  [LHC]    "4-bit computation from the start of Inkling 2 Small's pretraining", the paragraphs on
           fewer bits, on the backward pass and on communication.
  [4WEEK]  "Thinking Machines: Nvidia FP4 Up to 6x Faster, Runs Gain 8%", model-card update and
           "What Thinking Machines Changed".

Parity status of each function is stated in its docstring ("pinned by" names the tests).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_f32p = ctypes.POINTER(ctypes.c_float)
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle's C core."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        sig = {
            "orc_e2m1_rne_sat": (ctypes.c_uint32, [ctypes.c_float]),
            "orc_e2m1_value": (ctypes.c_float, [ctypes.c_uint32]),
            "orc_e4m3_rne_sat": (ctypes.c_uint32, [ctypes.c_float]),
            "orc_e4m3_value": (ctypes.c_float, [ctypes.c_uint32]),
            "orc_e8m0_value": (ctypes.c_float, [ctypes.c_uint32]),
            "orc_bf16_rne": (ctypes.c_uint32, [ctypes.c_float]),
            "orc_philox4x32_10": (None, [_u32p, _u32p, _u32p]),
            "orc_sr_word": (ctypes.c_uint32, [_u64, ctypes.c_uint32, _u64]),
            "orc_e4m3_sr": (ctypes.c_uint32, [ctypes.c_float, ctypes.c_uint32]),
            "orc_nvfp4_global_scales": (None, [ctypes.c_float, _f32p, _f32p]),
            "orc_nvfp4_quantize": (ctypes.c_int, [_f32p, _i64, _i64, _i64, _f32p, ctypes.c_int,
                                                  _u8p, _u8p, _f32p, _u8p]),
            "orc_nvfp4_dequantize": (None, [_u8p, _u8p, ctypes.c_float, _i64, _i64, _f32p]),
            "orc_mx_scale_exponent": (ctypes.c_int, [ctypes.c_float]),
            "orc_mxfp8_quantize_rows": (ctypes.c_int, [_f32p, _i64, _i64, ctypes.c_int, _u64,
                                                       ctypes.c_uint32, _u64, _u8p, _u8p]),
            "orc_mxfp8_dequantize_rows": (None, [_u8p, _u8p, _i64, _i64, _f32p]),
            "orc_mxfp8_requant_transpose": (ctypes.c_int, [_u8p, _u8p, _f32p, _i64, _i64, _i64,
                                                           ctypes.c_int, _u64, ctypes.c_uint32,
                                                           _u8p, _u8p]),
            "orc_fwht128": (None, [_f32p]),
            "orc_hadamard_scale": (ctypes.c_float, []),
            "orc_hadamard_rotate": (ctypes.c_int, [_f32p, _i64, _i64, _f32p]),
            "orc_hadamard_quant": (ctypes.c_int, [_f32p, _i64, _i64, ctypes.c_int, _u8p, _u8p,
                                                  _f32p]),
            "orc_hadamard_dequant": (ctypes.c_int, [_u8p, _u8p, ctypes.c_float, _i64, _i64,
                                                    _u16p]),
            "orc_hadamard_quant_mx": (ctypes.c_int, [_f32p, _i64, _i64, _u8p, _u8p]),
            "orc_hadamard_dequant_mx": (ctypes.c_int, [_u8p, _u8p, _i64, _i64, _u16p]),
            "orc_e2m1_rne_sat_range": (None, [ctypes.c_uint32, _u64, _u8p]),
            "orc_e4m3_rne_sat_range": (None, [ctypes.c_uint32, _u64, _u8p]),
            "orc_bf16_rne_array": (None, [_f32p, _i64, _u16p]),
            "orc_sr_words": (None, [_u64, ctypes.c_uint32, _u64, _i64, _u16p]),
            "orc_e4m3_sr_array": (None, [_f32p, _u16p, _i64, _u8p]),
            "orc_e4m3_rne_sat_array": (None, [_f32p, _i64, _u8p]),
            "orc_e2m1_rne_sat_array": (None, [_f32p, _i64, _u8p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(t)


# ----------------------------------------------------------------------------------------------
# bf16 <-> binary32 (exact widening; nearest-even narrowing)
# ----------------------------------------------------------------------------------------------
def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to binary32 exactly."""
    return (np.ascontiguousarray(h).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round binary32 to bf16 bit patterns, nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_rne_array(_p(x, _f32p), x.size, _p(out, _u16p))
    return out


# ----------------------------------------------------------------------------------------------
# Scalar formats (pinned by tests/test_oracle_formats.py: code tables, tie cases, saturation)
# ----------------------------------------------------------------------------------------------
def e2m1_rne_sat(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e2m1_rne_sat_array(_p(v, _f32p), v.size, _p(out, _u8p))
    return out


def e4m3_rne_sat(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_rne_sat_array(_p(v, _f32p), v.size, _p(out, _u8p))
    return out


def e2m1_value(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib().orc_e2m1_value(c) for c in range(16)], np.float32)
    return table[codes & 0xF]


def e4m3_value(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib().orc_e4m3_value(c) for c in range(256)], np.float32)
    return table[codes]


def e8m0_value(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    table = np.array([lib().orc_e8m0_value(c) for c in range(256)], np.float32)
    return table[b]


def e2m1_range(start: int, count: int) -> np.ndarray:
    """E2M1 codes of the binary32 bit patterns start .. start+count-1."""
    out = np.empty(count, np.uint8)
    lib().orc_e2m1_rne_sat_range(start, count, _p(out, _u8p))
    return out


def e4m3_range(start: int, count: int) -> np.ndarray:
    """E4M3 codes of the binary32 bit patterns start .. start+count-1."""
    out = np.empty(count, np.uint8)
    lib().orc_e4m3_rne_sat_range(start, count, _p(out, _u8p))
    return out


# ----------------------------------------------------------------------------------------------
# Philox and stochastic rounding (pinned by tests/test_oracle_philox_sr.py)
# ----------------------------------------------------------------------------------------------
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib().orc_philox4x32_10(_p(c, _u32p), _p(k, _u32p), _p(out, _u32p))
    return out


def sr_words(seed: int, stream_id: int, idx_base: int, n: int) -> np.ndarray:
    """The 16-bit stochastic-rounding numbers of output indices idx_base .. idx_base+n-1."""
    out = np.empty(n, np.uint16)
    lib().orc_sr_words(seed, stream_id, idx_base, n, _p(out, _u16p))
    return out


def e4m3_sr(v, r16) -> np.ndarray:
    """Stochastic rounding of binary32 v to E4M3 codes with 16-bit numbers r16 (one per value)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    r = np.ascontiguousarray(r16, dtype=np.uint16)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_sr_array(_p(v, _f32p), _p(r, _u16p), v.size, _p(out, _u8p))
    return out


# ----------------------------------------------------------------------------------------------
# NVFP4 with Four Over Six [LHC fewer-bits paragraph; DEBUT "Confirmed" list]
# (pinned by tests/test_oracle_nvfp4.py: exact-rational brute force of the 4/6 choice, 4.5 bits,
#  idempotence, worked cases)
# ----------------------------------------------------------------------------------------------
def nvfp4_global_scales(amax: float):
    ge, gd = ctypes.c_float(), ctypes.c_float()
    lib().orc_nvfp4_global_scales(float(amax), ctypes.byref(ge), ctypes.byref(gd))
    return np.float32(ge.value), np.float32(gd.value)


def nvfp4_quantize(x: np.ndarray, four_over_six: bool = True, amax=None, return_choice=False):
    """Quantise binary32 x of shape [rows, cols] or [nmat, rows, cols] (one per-tensor scale per
    matrix: per expert for weights).  Returns codes [.., rows, cols/2], sf [.., rows, cols/16],
    g_dec [nmat] (or a 0-d array for 2-D input), and optionally the 4/6 choice per block."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    squeeze = x.ndim == 2
    if squeeze:
        x = x[None]
    nmat, rows, cols = x.shape
    codes = np.empty((nmat, rows, cols // 2), np.uint8)
    sf = np.empty((nmat, rows, cols // 16), np.uint8)
    choice = np.empty((nmat, rows, cols // 16), np.uint8)
    g_dec = np.empty(nmat, np.float32)
    for m in range(nmat):
        am = None
        if amax is not None:
            am = np.array([np.asarray(amax, np.float32).reshape(-1)[m if np.size(amax) > 1 else 0]],
                          np.float32)
        gd = ctypes.c_float()
        rc = lib().orc_nvfp4_quantize(
            _p(x[m], _f32p), rows, cols, cols, None if am is None else _p(am, _f32p),
            int(bool(four_over_six)), _p(codes[m], _u8p), _p(sf[m], _u8p), ctypes.byref(gd),
            _p(choice[m], _u8p))
        if rc != 0:
            raise ValueError("nvfp4_quantize: cols must be a multiple of 16")
        g_dec[m] = gd.value
    if squeeze:
        codes, sf, choice, g_dec = codes[0], sf[0], choice[0], g_dec[0]
    if return_choice:
        return codes, sf, g_dec, choice
    return codes, sf, g_dec


def nvfp4_dequantize(codes: np.ndarray, sf: np.ndarray, g_dec) -> np.ndarray:
    """x_hat = (e2m1(q) * sf) * g_dec, for [rows, cols/2] or [nmat, rows, cols/2] codes."""
    codes = np.ascontiguousarray(codes, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    squeeze = codes.ndim == 2
    if squeeze:
        codes, sf = codes[None], sf[None]
    g = np.asarray(g_dec, np.float32).reshape(-1)
    nmat, rows, half = codes.shape
    cols = half * 2
    out = np.empty((nmat, rows, cols), np.float32)
    for m in range(nmat):
        lib().orc_nvfp4_dequantize(_p(codes[m], _u8p), _p(sf[m], _u8p), float(g[m]), rows, cols,
                                   _p(out[m], _f32p))
    return out[0] if squeeze else out


# ----------------------------------------------------------------------------------------------
# MXFP8 [LHC backward-pass paragraphs] (pinned by tests/test_oracle_mxfp8.py)
# ----------------------------------------------------------------------------------------------
def mx_scale_exponent(amax: float) -> int:
    return int(lib().orc_mx_scale_exponent(float(amax)))


def mxfp8_quantize_rows(z: np.ndarray, sr: bool, seed: int = 0, stream_id: int = 0,
                        idx_base: int = 0):
    """Quantise binary32 z[P, Q] along Q in 32-blocks.  Returns q [P, Q] (E4M3 codes) and
    e8 [P, Q/32]."""
    z = np.ascontiguousarray(z, np.float32)
    P, Q = z.shape
    q = np.empty((P, Q), np.uint8)
    e8 = np.empty((P, Q // 32), np.uint8)
    rc = lib().orc_mxfp8_quantize_rows(_p(z, _f32p), P, Q, int(bool(sr)), seed, stream_id,
                                       idx_base, _p(q, _u8p), _p(e8, _u8p))
    if rc != 0:
        raise ValueError("mxfp8: the blocked dimension must be a multiple of 32")
    return q, e8


def mxfp8_quantize(x: np.ndarray, colwise: bool, sr: bool = False, seed: int = 0,
                   stream_id: int = 0):
    """MXFP8 of binary32 x[R, C]: row-wise (blocks along C, output [R, C]) or column-wise (the
    transpose, blocks along R, output [C, R])."""
    z = np.ascontiguousarray(x.T if colwise else x, np.float32)
    return mxfp8_quantize_rows(z, sr, seed, stream_id)


def mxfp8_dequantize(q: np.ndarray, e8: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.uint8)
    e8 = np.ascontiguousarray(e8, np.uint8)
    squeeze = q.ndim == 2
    if squeeze:
        q, e8 = q[None], e8[None]
    n, P, Q = q.shape
    out = np.empty((n, P, Q), np.float32)
    for m in range(n):
        lib().orc_mxfp8_dequantize_rows(_p(q[m], _u8p), _p(e8[m], _u8p), P, Q, _p(out[m], _f32p))
    return out[0] if squeeze else out


def mxfp8_requant_transpose(codes, sf, g_dec, sr: bool = True, seed: int = 0, stream_id: int = 0):
    """Dequantise NVFP4 [.., rows, cols], transpose in binary32, requantise to MXFP8 along the new
    contiguous dimension.  Returns q_t [.., cols, rows] and e8_t [.., cols, rows/32]."""
    codes = np.ascontiguousarray(codes, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    squeeze = codes.ndim == 2
    if squeeze:
        codes, sf = codes[None], sf[None]
    nmat, rows, half = codes.shape
    cols = half * 2
    g = np.ascontiguousarray(np.asarray(g_dec, np.float32).reshape(-1))
    q_t = np.empty((nmat, cols, rows), np.uint8)
    e8_t = np.empty((nmat, cols, rows // 32), np.uint8)
    rc = lib().orc_mxfp8_requant_transpose(_p(codes, _u8p), _p(sf, _u8p), _p(g, _f32p), nmat,
                                           rows, cols, int(bool(sr)), seed, stream_id,
                                           _p(q_t, _u8p), _p(e8_t, _u8p))
    if rc != 0:
        raise ValueError("requant: rows must be a multiple of 32 and cols of 16")
    return (q_t[0], e8_t[0]) if squeeze else (q_t, e8_t)


# ----------------------------------------------------------------------------------------------
# Hadamard return-path codec [LHC communication paragraph] (pinned by tests/test_oracle_hadamard.py)
# ----------------------------------------------------------------------------------------------
def hadamard_scale() -> np.float32:
    return np.float32(lib().orc_hadamard_scale())


def fwht128(u: np.ndarray) -> np.ndarray:
    u = np.array(u, np.float32, copy=True).reshape(128)
    lib().orc_fwht128(_p(u, _f32p))
    return u


def hadamard_rotate(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty_like(x)
    if lib().orc_hadamard_rotate(_p(x, _f32p), x.shape[0], x.shape[1], _p(out, _f32p)) != 0:
        raise ValueError("hadamard: cols must be a multiple of 128")
    return out


def hadamard_quant(x: np.ndarray, four_over_six: bool = True):
    x = np.ascontiguousarray(x, np.float32)
    R, C = x.shape
    codes = np.empty((R, C // 2), np.uint8)
    sf = np.empty((R, C // 16), np.uint8)
    gd = ctypes.c_float()
    if lib().orc_hadamard_quant(_p(x, _f32p), R, C, int(bool(four_over_six)), _p(codes, _u8p),
                                _p(sf, _u8p), ctypes.byref(gd)) != 0:
        raise ValueError("hadamard: cols must be a multiple of 128")
    return codes, sf, np.float32(gd.value)


def hadamard_dequant(codes, sf, g_dec) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    R, half = codes.shape
    out = np.empty((R, half * 2), np.uint16)
    if lib().orc_hadamard_dequant(_p(codes, _u8p), _p(sf, _u8p), float(g_dec), R, half * 2,
                                  _p(out, _u16p)) != 0:
        raise ValueError("hadamard: cols must be a multiple of 128")
    return out


def hadamard_quant_mx(x: np.ndarray):
    """The 8.25-bit return-path codec: Hadamard(128) rotation, then MXFP8 (E4M3, E8M0 per 32,
    nearest-even).  Returns q [R, C] and e8 [R, C/32]."""
    x = np.ascontiguousarray(x, np.float32)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    e8 = np.empty((R, C // 32), np.uint8)
    if lib().orc_hadamard_quant_mx(_p(x, _f32p), R, C, _p(q, _u8p), _p(e8, _u8p)) != 0:
        raise ValueError("hadamard: cols must be a multiple of 128")
    return q, e8


def hadamard_dequant_mx(q, e8) -> np.ndarray:
    q = np.ascontiguousarray(q, np.uint8)
    e8 = np.ascontiguousarray(e8, np.uint8)
    R, C = q.shape
    out = np.empty((R, C), np.uint16)
    if lib().orc_hadamard_dequant_mx(_p(q, _u8p), _p(e8, _u8p), R, C, _p(out, _u16p)) != 0:
        raise ValueError("hadamard: cols must be a multiple of 128")
    return out


# ----------------------------------------------------------------------------------------------
# Routing, dispatch permutation, SwiGLU, combine, SGD.  The pages route each token to 8 of 384
# experts [4WEEK model-card update] and dispatch in NVFP4 [LHC communication paragraph]; they give
# no routing rule.  Readings: top-k of the logits (ties to the lower expert index), weights =
# softmax over the k chosen logits; rows grouped by expert, stable in (token, slot), each group
# zero-padded to a multiple of 128 rows.
# ----------------------------------------------------------------------------------------------
GROUP_PAD = 128


def route_topk(logits: np.ndarray, k: int):
    """idx int32 [T, k] (descending logit, ties to the lower expert index) and softmax weights
    over the chosen logits (float64 arithmetic, returned as binary32)."""
    logits = np.asarray(logits, np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    ex = np.exp(sel - sel[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def permute_plan(idx: np.ndarray, E: int, pad: int = GROUP_PAD):
    """Group offsets offs [E+1] (padded) and row_of [T, k]: the dispatched row of (token, slot)."""
    T, k = idx.shape
    counts = np.bincount(idx.reshape(-1), minlength=E)
    padded = (counts + pad - 1) // pad * pad
    offs = np.zeros(E + 1, np.int64)
    offs[1:] = np.cumsum(padded)
    row_of = np.empty((T, k), np.int64)
    fill = offs[:-1].copy()
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            row_of[t, j] = fill[e]
            fill[e] += 1
    return offs.astype(np.int32), row_of.astype(np.int32)


def permute_rows(src: np.ndarray, row_of: np.ndarray, rows_total: int) -> np.ndarray:
    """Gather row t of src into rows row_of[t, j]; other rows are zero."""
    out = np.zeros((rows_total,) + src.shape[1:], src.dtype)
    T, k = row_of.shape
    for t in range(T):
        for j in range(k):
            out[row_of[t, j]] = src[t]
    return out


def swiglu(gu: np.ndarray) -> np.ndarray:
    """h = silu(g) * u with g the first half of the columns and u the second half, in float64,
    returned as binary32 (the CUDA side rounds its binary32 result to bf16)."""
    gu = np.asarray(gu, np.float64)
    f = gu.shape[1] // 2
    g, u = gu[:, :f], gu[:, f:]
    return (g / (1.0 + np.exp(-g)) * u).astype(np.float32)


def swiglu_backward(gu: np.ndarray, dh: np.ndarray) -> np.ndarray:
    """Gradient of h = silu(g) * u: dg = dh * u * s * (1 + g * (1 - s)), du = dh * g * s with
    s = 1/(1+exp(-g)); float64, returned as binary32 [rows, 2f] (gate | up)."""
    gu = np.asarray(gu, np.float64)
    dh = np.asarray(dh, np.float64)
    f = gu.shape[1] // 2
    g, u = gu[:, :f], gu[:, f:]
    s = 1.0 / (1.0 + np.exp(-g))
    dg = dh * u * s * (1.0 + g * (1.0 - s))
    du = dh * g * s
    return np.concatenate([dg, du], axis=1).astype(np.float32)


def combine_backward(dy_bf16: np.ndarray, row_of: np.ndarray, w: np.ndarray, rows_total: int) -> np.ndarray:
    """dyhat[row_of[t, j]] = bf16(w[t, j] * dy[t]), one binary32 product per value; other rows 0."""
    dy = bf16_to_f32(dy_bf16)
    T, k = row_of.shape
    out = np.zeros((rows_total, dy.shape[1]), np.uint16)
    for j in range(k):
        out[row_of[:, j]] = f32_to_bf16((w[:, j:j + 1].astype(np.float32) * dy).astype(np.float32))
    return out


def combine(yhat_bf16: np.ndarray, row_of: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y[t] = sum over slots j in order of w[t, j] * yhat[row_of[t, j]]: one binary32 product and
    one binary32 add per slot, accumulator starting at 0; returned as bf16."""
    yh = bf16_to_f32(yhat_bf16)
    T, k = row_of.shape
    acc = np.zeros((T, yh.shape[1]), np.float32)
    for j in range(k):
        prod = (w[:, j:j + 1].astype(np.float32) * yh[row_of[:, j]]).astype(np.float32)
        acc = (acc + prod).astype(np.float32)
    return f32_to_bf16(acc)


def dispatch_backward(dxp_bf16: np.ndarray, row_of: np.ndarray) -> np.ndarray:
    """The gradient of the dispatch (row t of the tokens was sent to rows row_of[t, j]; the
    quantisation of the sent rows passes the gradient straight through): dx[t] = sum over slots j
    in order of dxp[row_of[t, j]], one binary32 add per slot from 0; returned as bf16."""
    g = bf16_to_f32(dxp_bf16)
    T, k = row_of.shape
    out = np.empty((T, g.shape[1]), np.uint16)
    for t in range(T):
        acc = np.zeros(g.shape[1], np.float32)
        for j in range(k):
            acc = (acc + g[row_of[t, j]]).astype(np.float32)
        out[t] = f32_to_bf16(acc)
    return out


def sgd_update(w32: np.ndarray, dw: np.ndarray, lr: float):
    """Plain SGD on the binary32 master weights (the pages keep master weights in FP32 but name
    no optimiser): w <- w - (lr * dw), one product and one difference; plus the bf16 copy that the
    next forward quantises."""
    step = (np.float32(lr) * np.asarray(dw, np.float32)).astype(np.float32)
    w_new = (np.asarray(w32, np.float32) - step).astype(np.float32)
    return w_new, f32_to_bf16(w_new)


# ----------------------------------------------------------------------------------------------
# Reference GEMMs: float64 products and sums of the dequantised operands (a library matmul as a
# step), rounded to binary32 at the end; S = sum of |a*b| gives the elementwise bound.
# ----------------------------------------------------------------------------------------------
def grouped_gemm_m(a_hat: np.ndarray, b_hat: np.ndarray, offs: np.ndarray, alpha=None):
    """M-grouped: rows offs[e]:offs[e+1] of A [R, K] times B[e] [N, K]^T -> D, S [R, N] (float64).
    Rows outside every group are zero."""
    R, K = a_hat.shape
    E, N, _ = b_hat.shape
    D = np.zeros((R, N), np.float64)
    S = np.zeros((R, N), np.float64)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        A = a_hat[lo:hi].astype(np.float64)
        B = b_hat[e].astype(np.float64)
        D[lo:hi] = A @ B.T
        S[lo:hi] = np.abs(A) @ np.abs(B).T
    return D, S


def grouped_gemm_k(a_hat: np.ndarray, b_hat: np.ndarray, offs: np.ndarray):
    """K-grouped: for each expert e, A[:, offs[e]:offs[e+1]] times B[:, same]^T -> D[e], S[e]
    of shape [M, N]; A is [M, R], B is [N, R] (float64)."""
    M, R = a_hat.shape
    N = b_hat.shape[0]
    E = len(offs) - 1
    D = np.zeros((E, M, N), np.float64)
    S = np.zeros((E, M, N), np.float64)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        A = a_hat[:, lo:hi].astype(np.float64)
        B = b_hat[:, lo:hi].astype(np.float64)
        D[e] = A @ B.T
        S[e] = np.abs(A) @ np.abs(B).T
    return D, S
