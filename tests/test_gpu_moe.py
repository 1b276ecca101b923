"""GPU parity of the MoE steps around the expert GEMMs: top-k routing (indices bit-exact, weights
to 1e-6 relative), the dispatch plan and the NVFP4 row gather (bit-exact), SwiGLU and its backward (within
one bf16 rounding: they call expf), the weighted combine and the SGD update of FP32 master weights (bit-exact).

Shapes: the small grouped MoE (8 experts, top-2) and the Inkling-shaped layer (384 experts, top-8,
N(0,1) logits plus a per-expert N(0,1) bias, 16384 tokens)."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import inputs, moe4
from gpu_helpers import DEV, empty_u8, first_mismatch, mma_layout, nvfp4_quantize, to_dev, to_np

pytestmark = pytest.mark.gpu


def _logits(T, E, bias, seed):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    if bias:
        lg = (lg + rng.standard_normal(E).astype(np.float32)).astype(np.float32)
    return lg


def _route_gpu(lg, k):
    T, E = lg.shape
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    moe4.moe4_route_topk(to_dev(lg), T, E, k, idx, w)
    torch.cuda.synchronize()
    return idx, w


@pytest.mark.parametrize("T,E,k,bias", [(4096, 8, 2, False), (16384, 384, 8, True), (33, 40, 32, False)])
def test_route_topk(T, E, k, bias):
    lg = _logits(T, E, bias, T + E)
    lg[0, :] = 0.25                          # a fully tied row: lowest expert indices win
    idx, w = _route_gpu(lg, k)
    ridx, rw = oracle.route_topk(lg, k)
    assert first_mismatch(to_np(idx), ridx) is None
    assert np.allclose(to_np(w), rw, rtol=1e-6, atol=0)


@pytest.mark.parametrize("T,E,k,bias", [(4096, 8, 2, False), (16384, 384, 8, True), (5, 3, 2, False)])
def test_permute_plan_and_gather(T, E, k, bias):
    lg = _logits(T, E, bias, 7 * T + E)
    ridx, _ = oracle.route_topk(lg, k)     # a seeded host input to both sides
    rows_cap = T * k + 127 * E
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_of = torch.empty((T, k), dtype=torch.int32, device=DEV)
    src_of = torch.empty(rows_cap, dtype=torch.int32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_PERMUTE_PLAN, T, k, E))
    moe4.moe4_permute_plan(to_dev(ridx), T, k, E, offs, row_of, src_of, rows_cap, ws)
    torch.cuda.synchronize()
    roffs, rrow = oracle.permute_plan(ridx, E)
    assert first_mismatch(to_np(offs), roffs) is None
    assert first_mismatch(to_np(row_of), rrow) is None
    Rp = int(roffs[-1])
    rsrc = np.full(rows_cap, -1, np.int32)
    rsrc[rrow.reshape(-1)] = np.repeat(np.arange(T, dtype=np.int32), k)
    assert first_mismatch(to_np(src_of), rsrc) is None
    # gather the NVFP4 rows of a token tensor
    cols = 256
    x = inputs.to_bf16_bits(np.random.default_rng(1).standard_normal((T, cols)).astype(np.float32))
    c, s, g = nvfp4_quantize(to_dev(x), 1, T, cols)
    oc, osf = empty_u8(Rp, cols // 2), empty_u8(Rp, cols // 16)
    moe4.moe4_permute_nvfp4(c, s, T, cols, src_of, Rp, oc, osf, 0)
    torch.cuda.synchronize()
    rc, rs, _ = oracle.nvfp4_quantize(oracle.bf16_to_f32(x))
    assert first_mismatch(to_np(oc), oracle.permute_rows(rc, rrow, Rp)) is None
    assert first_mismatch(to_np(osf), oracle.permute_rows(rs, rrow, Rp)) is None


def test_swiglu_within_one_bf16_ulp():
    rows, f = 640, 1024
    gu = (np.random.default_rng(2).standard_normal((rows, 2 * f)) * 4).astype(np.float32)
    h = torch.empty((rows, f), dtype=torch.int16, device=DEV)
    moe4.moe4_swiglu(to_dev(gu), rows, f, h)
    torch.cuda.synchronize()
    got = to_np(h, np.uint16).astype(np.int32)
    want = oracle.f32_to_bf16(oracle.swiglu(gu)).astype(np.int32)
    # bf16 bit patterns of same-sign values differ by the number of ulps between them
    assert np.max(np.abs(got - want)) <= 1


@pytest.mark.parametrize("rows,f", [(640, 1024), (0, 64), (160512, 2048)])
def test_swiglu_amax_equals_swiglu_and_max(rows, f):
    """moe4_swiglu_amax writes the same h as moe4_swiglu and the max |h| of those bf16 values
    (the last case is the 384-expert layer's H); an empty input gives amax 0."""
    gen = inputs.device_generator(13, rows, DEV)
    gu = inputs.device_normal((max(rows, 1), 2 * f), 3.0, gen, DEV, dtype=torch.float32)[:rows].contiguous()
    h0 = torch.empty((rows, f), dtype=torch.int16, device=DEV)
    h1 = torch.full((rows, f), -1, dtype=torch.int16, device=DEV)
    amax = torch.full((1,), -5.0, dtype=torch.float32, device=DEV)
    moe4.moe4_swiglu(gu, rows, f, h0)
    moe4.moe4_swiglu_amax(gu, rows, f, h1, amax)
    torch.cuda.synchronize()
    assert torch.equal(h0, h1)
    want = float(np.abs(oracle.bf16_to_f32(to_np(h0, np.uint16))).max()) if rows else 0.0
    assert float(to_np(amax)[0]) == want


def test_combine_bit_exact():
    T, k, d, R = 1000, 8, 512, 9000
    rng = np.random.default_rng(3)
    yh = inputs.to_bf16_bits(rng.standard_normal((R, d)).astype(np.float32))
    row_of = rng.permutation(R)[:T * k].reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    y = torch.empty((T, d), dtype=torch.int16, device=DEV)
    moe4.moe4_combine(to_dev(yh), to_dev(row_of), to_dev(w), T, k, d, y)
    torch.cuda.synchronize()
    assert first_mismatch(to_np(y, np.uint16), oracle.combine(yh, row_of, w)) is None


def test_dispatch_backward_bit_exact():
    """The gradient of the dispatch: each token's k dispatched rows summed in slot order, bit for
    bit against the oracle, on a top-8 plan over 384 experts (padding rows are never read)."""
    T, E, k, d = 2048, 384, 8, 512
    lg = _logits(T, E, True, 17)
    ridx, _ = oracle.route_topk(lg, k)
    roffs, rrow = oracle.permute_plan(ridx, E)
    R = int(roffs[-1])
    rng = np.random.default_rng(18)
    g = inputs.to_bf16_bits(rng.standard_normal((R, d)).astype(np.float32))
    dx = torch.empty((T, d), dtype=torch.int16, device=DEV)
    moe4.moe4_dispatch_backward(to_dev(g), to_dev(rrow), T, k, d, dx)
    torch.cuda.synchronize()
    assert first_mismatch(to_np(dx, np.uint16), oracle.dispatch_backward(g, rrow)) is None


def test_sgd_update_bit_exact():
    n = 1 << 16
    rng = np.random.default_rng(4)
    w32 = rng.standard_normal(n).astype(np.float32) * np.float32(0.02)
    dw = rng.standard_normal(n).astype(np.float32)
    wt = to_dev(w32)
    wb = torch.empty(n, dtype=torch.int16, device=DEV)
    moe4.moe4_sgd_update(wt, to_dev(dw), n, 1e-3, wb)
    torch.cuda.synchronize()
    rw, rb = oracle.sgd_update(w32, dw, 1e-3)
    assert first_mismatch(to_np(wt), rw) is None and first_mismatch(to_np(wb, np.uint16), rb) is None


def test_swiglu_backward_within_bf16_rounding():
    rows, f = 512, 1024
    rng = np.random.default_rng(5)
    gu = (rng.standard_normal((rows, 2 * f)) * 3).astype(np.float32)
    dh = rng.standard_normal((rows, f)).astype(np.float32)
    dgu = torch.empty((rows, 2 * f), dtype=torch.int16, device=DEV)
    moe4.moe4_swiglu_backward(to_dev(gu), to_dev(dh), rows, f, dgu)
    torch.cuda.synchronize()
    got = oracle.bf16_to_f32(to_np(dgu, np.uint16)).astype(np.float64)
    ref = oracle.swiglu_backward(gu, dh).astype(np.float64)
    # one bf16 rounding (2^-8 relative) plus a few binary32 ulps of the terms' size: near the zero
    # of silu' (g ~ -1.28) the factor 1 + g(1 - s) cancels in binary32
    g, u, d = gu[:, :f].astype(np.float64), gu[:, f:].astype(np.float64), dh.astype(np.float64)
    mag = np.abs(d) * (np.abs(u) * (1 + np.abs(g)) + np.abs(g))
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * np.concatenate([mag, mag], axis=1)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), int(bad.sum())


def _swiglu_bwd_mxfp8_both(gu, dh, rows, f):
    """Fused SwiGLU backward + MXFP8 (both layouts), and the unfused pair, on device tensors."""
    out = [empty_u8(rows, 2 * f), empty_u8(rows, 2 * f // 32), empty_u8(2 * f, rows), empty_u8(2 * f, rows // 32)]
    moe4.moe4_swiglu_backward_mxfp8(gu, dh, rows, f, *out)
    dgu = torch.empty((rows, 2 * f), dtype=torch.int16, device=DEV)
    moe4.moe4_swiglu_backward(gu, dh, rows, f, dgu)
    ref = [empty_u8(rows, 2 * f), empty_u8(rows, 2 * f // 32), empty_u8(2 * f, rows), empty_u8(2 * f, rows // 32)]
    moe4.mxfp8_quantize_rowcol(dgu, rows, 2 * f, *ref)
    torch.cuda.synchronize()
    return out, ref


@pytest.mark.parametrize("rows,f", [(96, 64), (512, 1024), (160512, 2048)])
def test_swiglu_backward_mxfp8_equals_unfused(rows, f):
    """Fused SwiGLU gradient + MXFP8 equals the SwiGLU gradient in bf16 followed by the row and
    transposed MXFP8 quantiser, byte for byte; the last case is the 384-expert layer's dGU."""
    gen = inputs.device_generator(9, rows, DEV)
    gu = inputs.device_normal((rows, 2 * f), 3.0, gen, DEV, dtype=torch.float32)
    dh = inputs.device_normal((rows, f), 1.0, gen, DEV, dtype=torch.float32)
    out, ref = _swiglu_bwd_mxfp8_both(gu, dh, rows, f)
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
    if rows % 128 == 0 and f % 64 == 0:
        mma = [empty_u8(rows, 2 * f), empty_u8(rows, 2 * f // 32), empty_u8(2 * f, rows), empty_u8(2 * f, rows // 32)]
        moe4.moe4_swiglu_backward_mxfp8(gu, dh, rows, f, *mma, flags=moe4.SF_OUT_MMA)
        torch.cuda.synchronize()
        assert torch.equal(mma[0], out[0]) and torch.equal(mma[2], out[2])
        assert torch.equal(mma[1].reshape(-1), mma_layout(out[1], rows, 2 * f // 32))
        assert torch.equal(mma[3].reshape(-1), mma_layout(out[3], 2 * f, rows // 32))


def test_swiglu_backward_mxfp8_against_oracle():
    """Dequantised row-wise output against the oracle's float64 SwiGLU gradient: the SwiGLU bound
    of the unfused test (one bf16 rounding, binary32 cancellation near the zero of silu') plus one
    E4M3 rounding of the bf16 value (2^-4 relative, or half the subnormal step of its block)."""
    rows, f = 256, 512
    rng = np.random.default_rng(15)
    gu = (rng.standard_normal((rows, 2 * f)) * 3).astype(np.float32)
    dh = rng.standard_normal((rows, f)).astype(np.float32)
    out, _ = _swiglu_bwd_mxfp8_both(to_dev(gu), to_dev(dh), rows, f)
    got = oracle.mxfp8_dequantize(to_np(out[0]), to_np(out[1])).astype(np.float64)
    ref = oracle.swiglu_backward(gu, dh).astype(np.float64)
    g, u, d = gu[:, :f].astype(np.float64), gu[:, f:].astype(np.float64), dh.astype(np.float64)
    mag = np.abs(d) * (np.abs(u) * (1 + np.abs(g)) + np.abs(g))
    tol = 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * np.concatenate([mag, mag], axis=1)
    blk_amax = (np.abs(ref) + tol).reshape(rows, 2 * f // 32, 32).max(axis=2)
    half_sub = np.repeat(2 * blk_amax / (448.0 * 1024), 32, axis=1)
    bound = tol + 2.0 ** -4 * (np.abs(ref) + tol) + half_sub
    bad = np.abs(got - ref) > bound
    assert not bad.any(), int(bad.sum())
    rq, re8 = oracle.mxfp8_quantize(oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))), colwise=True)
    assert np.mean(to_np(out[2]) == rq) >= 0.9  # the transposed layout: structure (same blocks)


@pytest.mark.parametrize("T,E,k,d", [(300, 16, 4, 96), (4096, 8, 2, 2048), (16384, 384, 8, 4096)])
def test_combine_backward_mxfp8_equals_unfused(T, E, k, d):
    """Fused combine gradient + MXFP8 (both layouts) equals moe4_combine_backward followed by
    mxfp8_quantize_rowcol, byte for byte; the last case is the 384-expert layer's dY."""
    lg = _logits(T, E, E > 8, 11 * T + E)
    ridx, rw = oracle.route_topk(lg, k)
    rows_cap = T * k + 127 * E
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_of = torch.empty((T, k), dtype=torch.int32, device=DEV)
    src_of = torch.empty(rows_cap, dtype=torch.int32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_PERMUTE_PLAN, T, k, E))
    moe4.moe4_permute_plan(to_dev(ridx), T, k, E, offs, row_of, src_of, rows_cap, ws)
    torch.cuda.synchronize()
    R = int(to_np(offs)[-1])
    dy = inputs.device_normal((T, d), 1.0, inputs.device_generator(12, T, DEV), DEV).view(torch.int16)
    w = to_dev(rw)
    out = [empty_u8(R, d), empty_u8(R, d // 32), empty_u8(d, R), empty_u8(d, R // 32)]
    moe4.moe4_combine_backward_mxfp8(dy, row_of, w, src_of, T, k, d, R, *out)
    dyhat = torch.empty((R, d), dtype=torch.int16, device=DEV)
    moe4.moe4_combine_backward(dy, row_of, w, src_of, T, k, d, R, dyhat)
    ref = [empty_u8(R, d), empty_u8(R, d // 32), empty_u8(d, R), empty_u8(d, R // 32)]
    moe4.mxfp8_quantize_rowcol(dyhat, R, d, *ref)
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
    if d % 128 == 0:
        # MOE4_SF_OUT_MMA: the scales as the library's layout change of the canonical ones
        mma = [empty_u8(R, d), empty_u8(R, d // 32), empty_u8(d, R), empty_u8(d, R // 32)]
        moe4.moe4_combine_backward_mxfp8(dy, row_of, w, src_of, T, k, d, R, *mma, flags=moe4.SF_OUT_MMA)
        torch.cuda.synchronize()
        assert torch.equal(mma[0], out[0]) and torch.equal(mma[2], out[2])
        assert torch.equal(mma[1].reshape(-1), mma_layout(out[1], R, d // 32))
        assert torch.equal(mma[3].reshape(-1), mma_layout(out[3], d, R // 32))


@pytest.mark.parametrize("T,E,k", [(4096, 8, 2), (300, 16, 4)])
def test_combine_backward_bit_exact(T, E, k):
    lg = _logits(T, E, True, 3 * T + E)
    ridx, rw = oracle.route_topk(lg, k)
    roffs, rrow = oracle.permute_plan(ridx, E)
    Rp = int(roffs[-1])
    rows_cap = T * k + 127 * E
    rsrc = np.full(rows_cap, -1, np.int32)
    rsrc[rrow.reshape(-1)] = np.repeat(np.arange(T, dtype=np.int32), k)
    d = 256
    dy = inputs.to_bf16_bits(np.random.default_rng(T).standard_normal((T, d)).astype(np.float32))
    out = torch.full((Rp, d), 0x7FC0, dtype=torch.int16, device=DEV)
    moe4.moe4_combine_backward(to_dev(dy), to_dev(rrow), to_dev(rw), to_dev(rsrc), T, k, d, Rp, out)
    torch.cuda.synchronize()
    assert first_mismatch(to_np(out, np.uint16), oracle.combine_backward(dy, rrow, rw, Rp)) is None


def test_permute_with_tensor_core_scale_layout():
    T, E, k, cols = 2000, 8, 2, 512
    lg = _logits(T, E, False, 99)
    ridx, _ = oracle.route_topk(lg, k)
    roffs, rrow = oracle.permute_plan(ridx, E)
    Rp = int(roffs[-1])
    rsrc = np.full(Rp, -1, np.int32)
    rsrc[rrow.reshape(-1)] = np.repeat(np.arange(T, dtype=np.int32), k)
    x = inputs.to_bf16_bits(np.random.default_rng(2).standard_normal((T, cols)).astype(np.float32))
    c, s, g = nvfp4_quantize(to_dev(x), 1, T, cols)
    oc, osf = empty_u8(Rp, cols // 2), empty_u8(Rp, cols // 16)
    moe4.moe4_permute_nvfp4(c, s, T, cols, to_dev(rsrc), Rp, oc, osf, moe4.SF_MMA_LAYOUT)
    torch.cuda.synchronize()
    rc, rs, _ = oracle.nvfp4_quantize(oracle.bf16_to_f32(x))
    want_s = oracle.permute_rows(rs, rrow, Rp)
    got = to_np(osf).reshape(-1)
    nblk = cols // 16
    r = np.arange(Rp)[:, None]
    b = np.arange(nblk)[None, :]
    off = ((r // 128) * (nblk // 4) + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4
    assert first_mismatch(got[off], want_s) is None
    assert first_mismatch(to_np(oc), oracle.permute_rows(rc, rrow, Rp)) is None
