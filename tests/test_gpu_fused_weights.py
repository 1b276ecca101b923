"""GPU parity of the fused weight path (nvfp4_quantize_f32_requant): FP32 master weights quantised
to NVFP4 with Four Over Six for the forward GEMM and, from those codes, dequantised, transposed and
requantised to MXFP8 with stochastic rounding for the backward GEMM ("4-bit computation from the
start of Inkling 2 Small's pretraining", lhc.media, backward-pass paragraphs; "Inkling 2 Small's
Native 4-Bit Training: Debut and Doubts", agihunt.info, "Confirmed": per-expert scales).

Bit for bit against the oracle on a ragged batched case, against the two separate entry points
(nvfp4_quantize_f32 with a given amax, then mxfp8_requant_transpose_sr) with both tile layouts and
at the layer's gate/up shape, and the skipping of experts that received no rows."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import inputs, moe4
from gpu_helpers import DEV, empty_u8, first_mismatch, to_dev, to_np

pytestmark = pytest.mark.gpu


def _amax_of_bf16(w32):
    return w32.to(torch.bfloat16).abs().reshape(w32.shape[0], -1).amax(dim=1).float().contiguous()


def _fused(w32, nmat, rows, cols, amax, seed, sid, flags, offs=None, fill=None):
    out = [empty_u8(nmat, rows, cols // 2), empty_u8(nmat * rows * cols // 16),
           torch.empty(nmat, dtype=torch.float32, device=DEV), empty_u8(nmat, cols, rows),
           empty_u8(nmat * cols * rows // 32)]
    if fill is not None:
        for t in out:
            t.view(torch.uint8).fill_(fill)
    moe4.nvfp4_quantize_f32_requant(w32, nmat, rows, cols, amax, out[0], out[1], out[2], out[3], out[4], seed, sid,
                                    offs, flags)
    torch.cuda.synchronize()
    return out


def _two_calls(w32, nmat, rows, cols, amax, seed, sid, flags):
    codes, sf = empty_u8(nmat, rows, cols // 2), empty_u8(nmat * rows * cols // 16)
    g = torch.empty(nmat, dtype=torch.float32, device=DEV)
    qflags = moe4.AMAX_GIVEN | (flags & (moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT))
    moe4.nvfp4_quantize_f32(w32, nmat, rows, cols, cols, codes, sf, g, amax, qflags)
    q, e8 = empty_u8(nmat, cols, rows), empty_u8(nmat * cols * rows // 32)
    rflags = flags & (moe4.SR | moe4.SF_MMA_LAYOUT | moe4.SF_OUT_MMA)
    moe4.mxfp8_requant_transpose_sr(codes, sf, g, nmat, rows, cols, q, e8, seed, sid, rflags)
    torch.cuda.synchronize()
    return [codes, sf, g, q, e8]


@pytest.mark.parametrize("sr", [True, False])
def test_fused_weight_path_against_oracle(sr):
    nmat, rows, cols = 3, 160, 192  # rows not a multiple of the 128-row tile
    rng = np.random.default_rng(31)
    w = (rng.standard_normal((nmat, rows, cols)) * 0.02 * np.exp2(rng.integers(-3, 4, (nmat, rows, 1))))
    w = w.astype(np.float32)
    w[1, :, :16] = 0.0  # all-zero blocks
    w32 = to_dev(w)
    amax = _amax_of_bf16(w32)
    seed, sid = 77, 3
    flags = moe4.FOUR_OVER_SIX | (moe4.SR if sr else 0)
    codes, sf, g, q, e8 = _fused(w32, nmat, rows, cols, amax, seed, sid, flags)
    wb = oracle.bf16_to_f32(oracle.f32_to_bf16(w))
    rc, rs, rg = oracle.nvfp4_quantize(wb, amax=to_np(amax))
    assert first_mismatch(to_np(codes).reshape(rc.shape), rc) is None
    assert first_mismatch(to_np(sf).reshape(rs.shape), rs) is None
    assert np.array_equal(to_np(g), rg)
    rq, re8 = oracle.mxfp8_requant_transpose(rc, rs, rg, sr=sr, seed=seed, stream_id=sid)
    assert first_mismatch(to_np(q).reshape(rq.shape), rq) is None
    assert first_mismatch(to_np(e8).reshape(re8.shape), re8) is None


def test_fused_weight_path_equals_two_calls_with_tile_layouts_and_skips():
    nmat, rows, cols = 6, 256, 512
    w32 = inputs.device_normal((nmat, rows, cols), 0.02, inputs.device_generator(31, 1, DEV), DEV,
                               dtype=torch.float32)
    amax = _amax_of_bf16(w32)
    flags = moe4.FOUR_OVER_SIX | moe4.SR | moe4.SF_MMA_LAYOUT | moe4.SF_OUT_MMA
    want = _two_calls(w32, nmat, rows, cols, amax, 5, 1, flags)
    got = _fused(w32, nmat, rows, cols, amax, 5, 1, flags)
    for a, b in zip(got, want):
        assert torch.equal(a, b)
    # experts 1 and 4 received no rows: their outputs are not written
    offs = to_dev(np.array([0, 128, 128, 384, 512, 512, 640], np.int32))
    got = _fused(w32, nmat, rows, cols, amax, 5, 1, flags, offs=offs, fill=0xA5)
    per = [rows * cols // 2, rows * cols // 16, 1, rows * cols, rows * cols // 32]
    for t, w_, n in zip(got, want, per):
        tv, wv = t.view(torch.uint8).reshape(nmat, -1), w_.view(torch.uint8).reshape(nmat, -1)
        for m in range(nmat):
            if m in (1, 4):
                assert bool((tv[m] == 0xA5).all())
            else:
                assert torch.equal(tv[m], wv[m])


def test_fused_weight_path_layer_shape():
    """The layer step's gate/up masters: 384 experts x [4096, 4096] FP32, against the two calls."""
    E, rows, cols = 384, 4096, 4096
    w32 = inputs.device_normal((E, rows, cols), 0.02, inputs.device_generator(31, 2, DEV), DEV, dtype=torch.float32)
    amax = _amax_of_bf16(w32)
    flags = moe4.FOUR_OVER_SIX | moe4.SR | moe4.SF_MMA_LAYOUT | moe4.SF_OUT_MMA
    got = _fused(w32, E, rows, cols, amax, 1003, 3, flags)
    want = _two_calls(w32, E, rows, cols, amax, 1003, 3, flags)
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_weight_path_chunked_on_two_streams_equals_one_call():
    """The layer step's schedule: the stack cut into expert chunks, chunk i+1's quantiser
    (MOE4_PASS_QUANT | MOE4_SHARE_SMS) on a side stream beside chunk i's requantiser
    (MOE4_PASS_REQUANT), each call on slices with its mat_base: every output byte equals one call
    over the whole stack, skipped experts included."""
    nmat, rows, cols = 10, 256, 512
    w32 = inputs.device_normal((nmat, rows, cols), 0.02, inputs.device_generator(31, 3, DEV), DEV,
                               dtype=torch.float32)
    amax = _amax_of_bf16(w32)
    offs = to_dev(np.array([0, 128, 128, 384, 512, 512, 640, 768, 768, 896, 1024], np.int32))
    flags = moe4.FOUR_OVER_SIX | moe4.SR | moe4.SF_MMA_LAYOUT | moe4.SF_OUT_MMA
    want = _fused(w32, nmat, rows, cols, amax, 9, 3, flags, offs=offs, fill=0x5A)
    out = [empty_u8(nmat, rows, cols // 2), empty_u8(nmat, rows * cols // 16),
           torch.empty(nmat, dtype=torch.float32, device=DEV), empty_u8(nmat, cols, rows),
           empty_u8(nmat, cols * rows // 32)]
    for t in out:
        t.view(torch.uint8).fill_(0x5A)
    bounds = [0, 3, 4, 7, 10]
    args = [(w32[a:b], b - a, rows, cols, amax[a:b], out[0][a:b], out[1][a:b], out[2][a:b], out[3][a:b],
             out[4][a:b], 9, 3, offs[a:b + 1]) for a, b in zip(bounds[:-1], bounds[1:])]
    side = torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    ev = [torch.cuda.Event() for _ in args]
    moe4.nvfp4_quantize_f32_requant(*args[0], flags | moe4.PASS_QUANT, mat_base=bounds[0])
    ev[0].record(cur)
    side.wait_event(ev[0])
    for i, a in enumerate(args):
        if i + 1 < len(args):
            moe4.nvfp4_quantize_f32_requant(*args[i + 1], flags | moe4.PASS_QUANT | moe4.SHARE_SMS, side,
                                            mat_base=bounds[i + 1])
            ev[i + 1].record(side)
        if i > 0:
            cur.wait_event(ev[i])
        moe4.nvfp4_quantize_f32_requant(*a, flags | moe4.PASS_REQUANT, mat_base=bounds[i])
    torch.cuda.synchronize()
    for a, b in zip(out, want):
        assert torch.equal(a.view(torch.uint8).reshape(-1), b.view(torch.uint8).reshape(-1))


def test_weight_path_slice_far_into_a_stack_against_oracle():
    """One matrix called as matrix 2^21 + 3 of a stack of [128, 256] matrices: its random indices
    start past 2^35 (the kernel's 64-bit index path) and equal the oracle's dequantise -> transpose
    -> MXFP8 rows with that index base."""
    rows, cols = 128, 256
    mat_base = (1 << 21) + 3
    rng = np.random.default_rng(32)
    w = (rng.standard_normal((1, rows, cols)) * 0.02).astype(np.float32)
    w32 = to_dev(w)
    amax = _amax_of_bf16(w32)
    flags = moe4.FOUR_OVER_SIX | moe4.SR
    codes, sf, g, q, e8 = [empty_u8(1, rows, cols // 2), empty_u8(1, rows * cols // 16),
                           torch.empty(1, dtype=torch.float32, device=DEV), empty_u8(1, cols, rows),
                           empty_u8(1, cols * rows // 32)]
    moe4.nvfp4_quantize_f32_requant(w32, 1, rows, cols, amax, codes, sf, g, q, e8, 21, 5, None, flags,
                                    mat_base=mat_base)
    torch.cuda.synchronize()
    wb = oracle.bf16_to_f32(oracle.f32_to_bf16(w))
    rc, rs, rg = oracle.nvfp4_quantize(wb, amax=to_np(amax))
    xt = np.ascontiguousarray(oracle.nvfp4_dequantize(rc, rs, rg)[0].T)
    rq, re8 = oracle.mxfp8_quantize_rows(xt, sr=True, seed=21, stream_id=5, idx_base=mat_base * cols * rows)
    assert first_mismatch(to_np(q).reshape(rq.shape), rq) is None
    assert first_mismatch(to_np(e8).reshape(re8.shape), re8) is None
