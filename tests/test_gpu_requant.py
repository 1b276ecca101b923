"""GPU parity of the MXFP8 requantise-transpose with stochastic rounding and of the MXFP8
quantiser of bf16 tensors, against the oracle, bit for bit ("4-bit computation from the start of
Inkling 2 Small's pretraining", lhc.media, backward-pass paragraphs).

Cases: several tiles with ragged edges (rows not a multiple of 128, columns not a multiple of 64),
batched matrices with one global random index, SR and nearest-even, several seeds and stream ids;
the backward-requant workload's full-size X [32768, 4096] (sampled output rows recomputed by the
oracle with the same global indices) and the SR unbiasedness check over seeds 0..15.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import inputs, moe4
from gpu_helpers import DEV, empty_u8, first_mismatch, mma_layout, nvfp4_quantize, to_dev, to_np

pytestmark = pytest.mark.gpu


def _requant_gpu(c, s, g, nmat, rows, cols, seed, sid, sr):
    q = empty_u8(nmat, cols, rows)
    e8 = empty_u8(nmat, cols, rows // 32)
    moe4.mxfp8_requant_transpose_sr(c, s, g, nmat, rows, cols, q, e8, seed, sid, moe4.SR if sr else 0)
    torch.cuda.synchronize()
    return q, e8


@pytest.mark.parametrize("shape", [(1, 32, 32), (1, 96, 96), (2, 160, 192), (3, 256, 512)])
@pytest.mark.parametrize("sr,seed,sid", [(True, 0, 0), (True, 12345, 7), (False, 0, 0)])
def test_requant_small(shape, sr, seed, sid):
    nmat, rows, cols = shape
    rng = np.random.default_rng(rows + cols + nmat)
    x = inputs.to_bf16_bits(rng.standard_t(3, (nmat * rows, cols)).astype(np.float32))
    c, s, g = nvfp4_quantize(to_dev(x), nmat, rows, cols)
    q, e8 = _requant_gpu(c, s, g, nmat, rows, cols, seed, sid, sr)
    oc, os_, og = oracle.nvfp4_quantize(oracle.bf16_to_f32(x).reshape(nmat, rows, cols))
    rq, re8 = oracle.mxfp8_requant_transpose(oc, os_, og, sr=sr, seed=seed, stream_id=sid)
    assert first_mismatch(to_np(e8), re8) is None
    assert first_mismatch(to_np(q), rq) is None


@pytest.mark.parametrize("sr", [True, False])
def test_requant_extreme_global_scales(sr):
    """Three matrices with global decode scales far apart: tiny (amax ~1e-36, g_dec below 2^-116),
    ordinary, and huge (amax ~1e30, g_dec above 2), the last two with all-zero 32-row blocks in
    some output rows (their block scale is the smallest, 2^-127)."""
    rows, cols = 160, 192
    rng = np.random.default_rng(77)
    base = rng.standard_t(3, (3, rows, cols))
    base[1:, :32, 5] = 0.0
    base[1:, 64:96, 70:74] = 0.0
    x = inputs.to_bf16_bits((base * np.array([1e-36, 1.0, 1e30])[:, None, None]).astype(np.float32))
    x = x.reshape(3 * rows, cols)
    c, s, g = nvfp4_quantize(to_dev(x), 3, rows, cols)
    q, e8 = _requant_gpu(c, s, g, 3, rows, cols, 5, 1, sr)
    oc, os_, og = oracle.nvfp4_quantize(oracle.bf16_to_f32(x).reshape(3, rows, cols))
    assert og[0] < 2.0 ** -116 and og[2] > 2.0
    rq, re8 = oracle.mxfp8_requant_transpose(oc, os_, og, sr=sr, seed=5, stream_id=1)
    assert first_mismatch(to_np(e8), re8) is None
    assert first_mismatch(to_np(q), rq) is None


def test_requant_single_expert_operands():
    rng = inputs.host_rng(1, 0)
    x = inputs.to_bf16_bits(inputs.host_outliers(rng, inputs.host_normal(rng, (256, 512))))
    w = inputs.to_bf16_bits(inputs.host_normal(inputs.host_rng(1, 1), (256, 512), 0.02))
    for t, sid in ((x, 0), (w, 1)):
        c, s, g = nvfp4_quantize(to_dev(t), 1, 256, 512)
        q, e8 = _requant_gpu(c, s, g, 1, 256, 512, 0, sid, True)
        oc, os_, og = oracle.nvfp4_quantize(oracle.bf16_to_f32(t))
        rq, re8 = oracle.mxfp8_requant_transpose(oc, os_, og, sr=True, seed=0, stream_id=sid)
        assert first_mismatch(to_np(q), rq) is None and first_mismatch(to_np(e8), re8) is None


def test_requant_full_size_x_sampled_output_rows():
    rows, cols = 32768, 4096
    x = inputs.device_student_t((rows, cols), inputs.device_generator(4, 0, DEV), DEV).view(torch.int16)
    c, s, g = nvfp4_quantize(x, 1, rows, cols)
    seed, sid = 3, 2
    q, e8 = _requant_gpu(c, s, g, 1, rows, cols, seed, sid, True)
    qn, e8n = to_np(q)[0], to_np(e8)[0]
    x32 = oracle.bf16_to_f32(to_np(x, np.uint16))
    amax = np.abs(x32).max()
    for c0 in [0, 1024, 4064]:                 # 32 output rows starting at c0
        # the oracle quantises the 32 input columns itself (16-blocks never straddle the slice)
        codes, scl, gd = oracle.nvfp4_quantize(np.ascontiguousarray(x32[:, c0:c0 + 32]), amax=amax)
        xh = oracle.nvfp4_dequantize(codes, scl, gd)               # [rows, 32]
        rq, re8 = oracle.mxfp8_quantize_rows(np.ascontiguousarray(xh.T), sr=True, seed=seed, stream_id=sid,
                                             idx_base=c0 * rows)
        assert first_mismatch(qn[c0:c0 + 32], rq) is None
        assert first_mismatch(e8n[c0:c0 + 32], re8) is None


def test_sr_unbiased_over_seeds_on_device():
    rows, cols = 1024, 512
    x = inputs.to_bf16_bits(np.random.default_rng(8).standard_t(3, (rows, cols)).astype(np.float32))
    c, s, g = nvfp4_quantize(to_dev(x), 1, rows, cols)
    xh = oracle.nvfp4_dequantize(*oracle.nvfp4_quantize(oracle.bf16_to_f32(x))).T.astype(np.float64)
    acc = np.zeros_like(xh)
    for seed in range(16):
        q, e8 = _requant_gpu(c, s, g, 1, rows, cols, seed, 0, True)
        acc += oracle.mxfp8_dequantize(to_np(q)[0], to_np(e8)[0])
    mean = acc / 16
    _, er = oracle.mxfp8_requant_transpose(*oracle.nvfp4_quantize(oracle.bf16_to_f32(x)), sr=False)
    scale = np.repeat(np.exp2(er.astype(np.float64) - 127), 32, axis=1)
    grid = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    v = np.abs(xh) / scale
    lo = np.clip(np.searchsorted(grid, v, side="right") - 1, 0, 125)
    ulp = (grid[lo + 1] - grid[lo]) * scale
    p = np.clip((np.abs(xh) - grid[lo] * scale) / ulp, 0, 1)
    sd = ulp * np.sqrt(p * (1 - p) / 16)
    live = sd > 0
    z = ((mean - xh)[live] / sd[live]).sum() / np.sqrt(live.sum())
    assert abs(z) < 5, z


@pytest.mark.parametrize("layout", ["row", "col"])
@pytest.mark.parametrize("sr", [False, True])
def test_mxfp8_quantize(layout, sr):
    rows, cols = 320, 192
    rng = np.random.default_rng(11)
    x = inputs.to_bf16_bits((rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-6, 6, (rows, 1))))
                            .astype(np.float32))
    shape_q = (rows, cols) if layout == "row" else (cols, rows)
    q = empty_u8(*shape_q)
    e8 = empty_u8(shape_q[0], shape_q[1] // 32)
    flags = (moe4.ROWWISE if layout == "row" else moe4.COLWISE) | (moe4.SR if sr else 0)
    moe4.mxfp8_quantize(to_dev(x), rows, cols, q, e8, 77, 4, flags)
    torch.cuda.synchronize()
    rq, re8 = oracle.mxfp8_quantize(oracle.bf16_to_f32(x), colwise=(layout == "col"), sr=sr, seed=77, stream_id=4)
    assert first_mismatch(to_np(q), rq) is None and first_mismatch(to_np(e8), re8) is None


@pytest.mark.parametrize("shape", [(320, 192), (96, 96), (160512 // 4, 4096)])
def test_mxfp8_quantize_rowcol(shape):
    """Both layouts from one read equal the oracle's row-wise and transposed MXFP8 (nearest-even);
    the last case is a quarter of the backward's dY at the 384-expert layer, checked on sampled rows
    and columns."""
    rows, cols = shape
    rng = np.random.default_rng(rows)
    x = inputs.to_bf16_bits((rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-6, 6, (rows, 1))))
                            .astype(np.float32))
    x[:32] = 0  # an all-zero block in both layouts
    qr, er = empty_u8(rows, cols), empty_u8(rows, cols // 32)
    qc, ec = empty_u8(cols, rows), empty_u8(cols, rows // 32)
    moe4.mxfp8_quantize_rowcol(to_dev(x), rows, cols, qr, er, qc, ec)
    torch.cuda.synchronize()
    xf = oracle.bf16_to_f32(x)
    if rows * cols <= 1 << 20:
        rq, re8 = oracle.mxfp8_quantize(xf, colwise=False)
        assert first_mismatch(to_np(qr), rq) is None and first_mismatch(to_np(er), re8) is None
        rq, re8 = oracle.mxfp8_quantize(xf, colwise=True)
        assert first_mismatch(to_np(qc), rq) is None and first_mismatch(to_np(ec), re8) is None
        return
    pick = np.random.default_rng(1).choice(rows, 64, replace=False)
    rq, re8 = oracle.mxfp8_quantize(xf[pick], colwise=False)
    assert first_mismatch(to_np(qr)[pick], rq) is None and first_mismatch(to_np(er)[pick], re8) is None
    pickc = np.random.default_rng(2).choice(cols, 16, replace=False)
    rq, re8 = oracle.mxfp8_quantize(np.ascontiguousarray(xf[:, pickc]), colwise=True)
    assert first_mismatch(to_np(qc)[pickc], rq) is None and first_mismatch(to_np(ec)[pickc], re8) is None


def test_requant_reads_tensor_core_scale_layout():
    nmat, rows, cols = 2, 256, 512
    rng = np.random.default_rng(31)
    x = inputs.to_bf16_bits(rng.standard_t(3, (nmat * rows, cols)).astype(np.float32))
    xd = to_dev(x)
    c, s, g = nvfp4_quantize(xd, nmat, rows, cols)
    c2, s2, g2 = nvfp4_quantize(xd, nmat, rows, cols, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT)
    q1, e1 = _requant_gpu(c, s, g, nmat, rows, cols, 5, 1, True)
    q2 = empty_u8(nmat, cols, rows)
    e2 = empty_u8(nmat, cols, rows // 32)
    moe4.mxfp8_requant_transpose_sr(c2, s2, g2, nmat, rows, cols, q2, e2, 5, 1, moe4.SR | moe4.SF_MMA_LAYOUT)
    torch.cuda.synchronize()
    oc, os_, og = oracle.nvfp4_quantize(oracle.bf16_to_f32(x).reshape(nmat, rows, cols))
    rq, re8 = oracle.mxfp8_requant_transpose(oc, os_, og, sr=True, seed=5, stream_id=1)
    assert first_mismatch(to_np(q2), rq) is None and first_mismatch(to_np(e2), re8) is None
    assert torch.equal(q1, q2) and torch.equal(e1, e2)


@pytest.mark.parametrize("sr", [True, False])
def test_requant_scales_in_tile_layout(sr):
    """MOE4_SF_OUT_MMA: the same codes, and the scales as moe4_sf_to_mma_layout of the canonical
    ones (the canonical output has its own parity tests); two matrices, so tiles of the scale
    matrix [nmat * cols, rows / 32] follow on across the matrix boundary."""
    nmat, rows, cols = 2, 384, 256
    rng = np.random.default_rng(91)
    x = inputs.to_bf16_bits(rng.standard_t(3, (nmat * rows, cols)).astype(np.float32))
    c, s, g = nvfp4_quantize(to_dev(x), nmat, rows, cols)
    base = moe4.SR if sr else 0
    q0, e0 = _requant_gpu(c, s, g, nmat, rows, cols, 9, 2, sr)
    q1, e1 = empty_u8(nmat, cols, rows), empty_u8(nmat, cols, rows // 32)
    moe4.mxfp8_requant_transpose_sr(c, s, g, nmat, rows, cols, q1, e1, 9, 2, base | moe4.SF_OUT_MMA)
    torch.cuda.synchronize()
    assert torch.equal(q0, q1)
    assert torch.equal(e1.reshape(-1), mma_layout(e0, nmat * cols, rows // 32))


def test_rowcol_scales_in_tile_layout():
    rows, cols = 384, 256
    x = inputs.device_student_t((rows, cols), inputs.device_generator(92, 0, DEV), DEV).view(torch.int16)
    ref = [empty_u8(rows, cols), empty_u8(rows, cols // 32), empty_u8(cols, rows), empty_u8(cols, rows // 32)]
    moe4.mxfp8_quantize_rowcol(x, rows, cols, *ref)
    out = [empty_u8(rows, cols), empty_u8(rows, cols // 32), empty_u8(cols, rows), empty_u8(cols, rows // 32)]
    moe4.mxfp8_quantize_rowcol(x, rows, cols, *out, flags=moe4.SF_OUT_MMA)
    torch.cuda.synchronize()
    assert torch.equal(out[0], ref[0]) and torch.equal(out[2], ref[2])
    assert torch.equal(out[1].reshape(-1), mma_layout(ref[1], rows, cols // 32))
    assert torch.equal(out[3].reshape(-1), mma_layout(ref[3], cols, rows // 32))


@pytest.mark.parametrize("sr", [True, False])
def test_requant_rows_of_very_different_scale(sr):
    """Every seventh input row is 10^-4 times smaller: its NVFP4 block scales sit more than 2^10
    below the others in the same tile, so after the MXFP8 scaling some of its values fall below
    2^-6 and round into the E4M3 subnormals (the per-value path of the stochastic rounding);
    tiles without such rows take the tile-wide fast path."""
    nmat, rows, cols = 2, 256, 128
    rng = np.random.default_rng(71)
    base = rng.standard_t(3, (nmat, rows, cols))
    base[:, ::7, :] *= 1e-4
    x = inputs.to_bf16_bits(base.astype(np.float32)).reshape(nmat * rows, cols)
    c, s, g = nvfp4_quantize(to_dev(x), nmat, rows, cols)
    q, e8 = _requant_gpu(c, s, g, nmat, rows, cols, 11, 3, sr)
    oc, os_, og = oracle.nvfp4_quantize(oracle.bf16_to_f32(x).reshape(nmat, rows, cols))
    rq, re8 = oracle.mxfp8_requant_transpose(oc, os_, og, sr=sr, seed=11, stream_id=3)
    sub = ((rq & 0x78) == 0) & ((rq & 0x07) != 0)
    assert sub.sum() > 1000  # the E4M3 subnormal range is exercised
    assert first_mismatch(to_np(e8), re8) is None
    assert first_mismatch(to_np(q), rq) is None


def test_requant_full_size_gate_up_weights_sampled():
    """The layer step's largest requantisation as it runs there: 384 experts' gate/up weights
    [384, 4096, 4096] N(0, 0.02), NVFP4 with per-expert scales in the tile layout, to MXFP8
    [384, 4096, 4096] transposed with stochastic rounding (6.4G values: 32-bit Philox counters).
    Sampled: experts 0, 191 and 383, three slices of 32 output rows each; the oracle quantises
    those input columns with the expert's amax and rounds them with the global output index."""
    E, rows, cols = 384, 4096, 4096
    w = inputs.device_normal((E * rows, cols), 0.02, inputs.device_generator(22, 0, DEV), DEV).view(torch.int16)
    c, s, g = nvfp4_quantize(w, E, rows, cols, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT)
    q, e8 = empty_u8(E, cols, rows), empty_u8(E, cols, rows // 32)
    seed, sid = 7, 3
    moe4.mxfp8_requant_transpose_sr(c, s, g, E, rows, cols, q, e8, seed, sid, moe4.SR | moe4.SF_MMA_LAYOUT)
    torch.cuda.synchronize()
    del c, s
    for e in [0, 191, 383]:
        we = oracle.bf16_to_f32(to_np(w[e * rows:(e + 1) * rows], np.uint16))
        amax = np.abs(we).max()
        qn, e8n = to_np(q[e]), to_np(e8[e])
        for c0 in [0, 2048, 4064]:
            codes, scl, gd = oracle.nvfp4_quantize(np.ascontiguousarray(we[:, c0:c0 + 32]), amax=amax)
            assert np.asarray(gd).reshape(-1)[0] == to_np(g)[e]
            xh = oracle.nvfp4_dequantize(codes, scl, gd)
            rq, re8 = oracle.mxfp8_quantize_rows(np.ascontiguousarray(xh.T), sr=True, seed=seed, stream_id=sid,
                                                 idx_base=(e * cols + c0) * rows)
            assert first_mismatch(qn[c0:c0 + 32], rq) is None
            assert first_mismatch(e8n[c0:c0 + 32], re8) is None


def test_mxfp8_colwise_sr_beyond_2_35_values():
    """More than 2^35 output values (131072 x 262400): with eight values per Philox call the
    counter's second word becomes non-zero for the last output rows, so the transposing kernel
    runs its 64-bit counter instance.  Input: bf16 values from a multiplicative hash of the
    element index (all finite); checked on the first and the last 32 output rows against the
    oracle with the global index."""
    rows, cols = 131072, 262400
    n = rows * cols
    assert n > (1 << 35)
    x = torch.empty(n, dtype=torch.int16, device=DEV)
    step = 1 << 28
    for s0 in range(0, n, step):
        i = torch.arange(s0, min(n, s0 + step), device=DEV, dtype=torch.int64)
        h = (i * 2654435761) & 0xFFFFFFFF
        bits = 0x3C00 + ((h >> 7) & 0x07FF) + ((h >> 20) & 1) * 0x8000
        x[s0:s0 + len(i)] = bits.to(torch.int32).to(torch.int16)
        del i, h, bits
    q, e8 = empty_u8(cols, rows), empty_u8(cols, rows // 32)
    seed, sid = 9, 5
    moe4.mxfp8_quantize(x, rows, cols, q, e8, seed, sid, moe4.COLWISE | moe4.SR)
    torch.cuda.synchronize()
    xv = x.view(rows, cols)
    for c0 in [0, cols - 32]:
        xs = oracle.bf16_to_f32(to_np(xv[:, c0:c0 + 32].contiguous(), np.uint16))
        rq, re8 = oracle.mxfp8_quantize_rows(np.ascontiguousarray(xs.T), sr=True, seed=seed, stream_id=sid,
                                             idx_base=c0 * rows)
        assert c0 == 0 or (c0 * rows) // 8 >= (1 << 32)  # the last slice: counter word 1 is 1
        assert first_mismatch(to_np(q[c0:c0 + 32]), rq) is None
        assert first_mismatch(to_np(e8[c0:c0 + 32]), re8) is None


def test_sr_unbiased_over_seeds_backward_requant_shape():
    """The backward-requant workload's activations, X [32768, 4096] Student-t(3): NVFP4, then the
    MXFP8 stochastic-rounding transpose with seeds 0..15 ("4-bit computation from the start of
    Inkling 2 Small's pretraining", backward-pass paragraphs: the value is kept on average).  Over
    the 134M outputs, the mean of the 16 decoded draws minus the exact NVFP4 value, in units of
    each value's predicted standard deviation, aggregates to |z| < 5, both plainly and signed by
    the value.  The signed statistic sees a pull toward zero: with fractions spread evenly over a
    gap, a deficit of b gaps per value moves it by about b * 4 * pi * sqrt(n), so 8-bit random
    numbers (b = 2^-9 on average) would give about -285 here and the 16-bit ones (b = 2^-17)
    about -1.1.  The codes and scales are the oracle's bit for bit in the other tests; this
    checks the statistics at full size."""
    rows, cols = 32768, 4096
    x = inputs.device_student_t((rows, cols), inputs.device_generator(4, 7, DEV), DEV).view(torch.int16)
    c, s, g = nvfp4_quantize(x, 1, rows, cols)
    # the exact binary32 values the requantiser rounds, from the oracle's decode, transposed
    xh = oracle.nvfp4_dequantize(to_np(c)[0], to_np(s)[0], float(to_np(g)[0])).T
    xh = torch.from_numpy(np.ascontiguousarray(xh)).to(DEV).double()
    e4 = torch.from_numpy(oracle.e4m3_value(np.arange(256, dtype=np.uint8) & 0x7F).astype(np.float64)).to(DEV)
    e4 = torch.where(torch.arange(256, device=DEV) >= 128, -e4, e4)
    acc = torch.zeros_like(xh)
    e8_first = None
    for seed in range(16):
        q, e8 = _requant_gpu(c, s, g, 1, rows, cols, seed, 0, True)
        q, e8 = q[0], e8[0]
        if e8_first is None:
            e8_first = e8.clone()
        assert torch.equal(e8, e8_first)  # the scales do not depend on the random numbers
        scale = torch.exp2(e8.double() - 127).repeat_interleave(32, dim=1)
        acc += e4[q.long()] * scale
        del q
    mean = acc / 16
    scale = torch.exp2(e8_first.double() - 127).repeat_interleave(32, dim=1)
    grid = torch.from_numpy(oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)).to(DEV)
    v = xh.abs() / scale
    lo = (torch.searchsorted(grid, v.reshape(-1), right=True) - 1).clamp(0, 125).reshape(v.shape)
    gap = (grid[lo + 1] - grid[lo]) * scale
    p = ((xh.abs() - grid[lo] * scale) / gap).clamp(0, 1)
    sd = gap * torch.sqrt(p * (1 - p) / 16)
    live = sd > 0
    z = (mean - xh)[live] / sd[live]
    n = float(live.sum())
    z_plain = float(z.sum()) / np.sqrt(n)
    z_signed = float((z * torch.sign(xh[live])).sum()) / np.sqrt(n)
    assert n > 1e8
    assert abs(z_plain) < 5 and abs(z_signed) < 5, (z_plain, z_signed)
