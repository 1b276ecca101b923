"""GPU parity of the NVFP4 quantiser (Four Over Six), the dequantiser, the Hadamard codec and the
device's own conversions, against the oracle, bit for bit.

Inputs follow the seeded recipe of precision_moe_numerics_03_b300.inputs: the single-expert
workload (X 256x512 N(0,1) with 1% outliers x20, W 512x256 N(0, 0.02)), ragged shapes, batched
per-expert matrices, degenerate tensors, and the backward-requant workload's full-size X
[32768, 4096] Student-t(3) and W [384, 2048, 4096] N(0, 0.02) with sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import inputs, moe4
from gpu_helpers import DEV, empty_u8, first_mismatch, nvfp4_quantize, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    moe4.load()


def _check_quant(x_bits_np, nmat, rows, cols, fos=True, amax=None):
    x32 = oracle.bf16_to_f32(x_bits_np).reshape(nmat, rows, cols)
    c, s, g = nvfp4_quantize(to_dev(x_bits_np.reshape(nmat * rows, cols)), nmat, rows, cols,
                             moe4.FOUR_OVER_SIX if fos else 0, amax=amax)
    rc, rs, rg = oracle.nvfp4_quantize(x32, four_over_six=fos, amax=amax)
    msg = first_mismatch(to_np(c), rc) or first_mismatch(to_np(s), rs) or first_mismatch(to_np(g), rg)
    assert msg is None, msg
    return c, s, g


def _single_expert():
    rng = inputs.host_rng(1, 0)
    x = inputs.host_outliers(rng, inputs.host_normal(rng, (256, 512)))
    w = inputs.host_normal(inputs.host_rng(1, 1), (256, 512), 0.02)
    return inputs.to_bf16_bits(x), inputs.to_bf16_bits(w)


@pytest.mark.parametrize("fos", [True, False])
def test_single_expert_operands(fos):
    x, w = _single_expert()
    _check_quant(x, 1, 256, 512, fos)
    _check_quant(w, 1, 256, 512, fos)


@pytest.mark.parametrize("shape", [(1, 1, 16), (1, 3, 48), (1, 300, 144), (3, 37, 256), (5, 128, 64)])
def test_ragged_and_batched(shape):
    nmat, rows, cols = shape
    rng = np.random.default_rng(rows * 7 + cols)
    x = rng.standard_t(3, (nmat, rows, cols)).astype(np.float32)
    x *= np.exp2(rng.integers(-8, 8, (nmat, 1, 1))).astype(np.float32)  # per-matrix scale
    _check_quant(inputs.to_bf16_bits(x), nmat, rows, cols)


def test_amax_given_and_strided_rows():
    rng = np.random.default_rng(3)
    rows, cols, ld = 64, 96, 128
    full = inputs.to_bf16_bits(rng.standard_normal((rows, ld)).astype(np.float32))
    x = full[:, :cols]
    amax = np.float32(7.25)
    c, s, g = nvfp4_quantize(to_dev(full), 1, rows, cols, amax=amax, ld=ld)
    rc, rs, rg = oracle.nvfp4_quantize(oracle.bf16_to_f32(np.ascontiguousarray(x)), amax=amax)
    assert first_mismatch(to_np(c)[0], rc) is None and first_mismatch(to_np(s)[0], rs) is None
    assert to_np(g)[0] == rg


def test_degenerate_tensors():
    z = np.zeros((4, 32), np.uint16)
    _check_quant(z, 1, 4, 32)                                   # amax 0: g_dec = 1, all codes 0
    neg = inputs.to_bf16_bits(-np.zeros((2, 32), np.float32))
    _check_quant(neg, 1, 2, 32)                                 # -0 keeps its sign
    tiny = inputs.to_bf16_bits(np.full((2, 32), 1e-39, np.float32))
    _check_quant(tiny, 1, 2, 32)                                # g_enc overflows to FLT_MAX
    big = inputs.to_bf16_bits(np.array([[3e38] + [1.0] * 15], np.float32))
    _check_quant(big, 1, 1, 16)
    # no rows: only g_dec is written (1.0)
    c, s, g = nvfp4_quantize(torch.empty((0, 32), dtype=torch.int16, device=DEV), 2, 0, 32)
    assert list(to_np(g)) == [1.0, 1.0]


@pytest.mark.parametrize("rows,cols", [(256, 512), (384, 192), (128, 320), (256, 448)])
def test_sf_mma_layout_is_a_permutation(rows, cols):
    """The tile-layout scale offsets divide the block index by cols/64 through a multiply and
    shift: cols/64 = 8, 3, 5 and 7 here."""
    rng = np.random.default_rng(4)
    nmat = 2
    x = inputs.to_bf16_bits(rng.standard_normal((nmat * rows, cols)).astype(np.float32))
    xd = to_dev(x)
    c0, s0, g0 = nvfp4_quantize(xd, nmat, rows, cols)
    c1, s1, g1 = nvfp4_quantize(xd, nmat, rows, cols, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT)
    out = empty_u8(nmat, rows, cols // 16)
    moe4.moe4_sf_to_mma_layout(s0, nmat, rows, cols // 16, out)
    torch.cuda.synchronize()
    assert torch.equal(c0, c1) and torch.equal(g0, g1) and torch.equal(out, s1)
    # the layout itself, recomputed on the host for every byte
    s0n, s1n = to_np(s0), to_np(s1).reshape(nmat, -1)
    nblk = cols // 16
    for m in range(nmat):
        for r in range(0, rows, 37):
            for b in range(nblk):
                off = ((r // 128) * (nblk // 4) + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4
                assert s1n[m, off] == s0n[m, r, b]


@pytest.mark.parametrize("bf16_out", [True, False])
def test_dequantize(bf16_out):
    x, _ = _single_expert()
    c, s, g = nvfp4_quantize(to_dev(x), 1, 256, 512)
    out = torch.empty((1, 256, 512), dtype=torch.int16 if bf16_out else torch.float32, device=DEV)
    moe4.nvfp4_dequantize(c, s, g, 1, 256, 512, out, moe4.OUT_BF16 if bf16_out else moe4.OUT_F32)
    torch.cuda.synchronize()
    ref = oracle.nvfp4_dequantize(*oracle.nvfp4_quantize(oracle.bf16_to_f32(x)))
    if bf16_out:
        assert first_mismatch(to_np(out, np.uint16)[0], oracle.f32_to_bf16(ref)) is None
    else:
        assert first_mismatch(to_np(out)[0], ref) is None


def test_requant_stream_x_full_size_sampled_rows():
    rows, cols = 32768, 4096
    g = inputs.device_generator(4, 0, DEV)
    x = inputs.device_student_t((rows, cols), g, DEV)
    xb = x.view(torch.int16)
    c, s, gd = nvfp4_quantize(xb, 1, rows, cols)
    host = to_np(xb, np.uint16)
    amax = np.abs(oracle.bf16_to_f32(host)).max()
    sample = np.random.default_rng(0).choice(rows, 64, replace=False)
    sample = np.concatenate([sample, [0, rows - 1]])
    rc, rs, rg = oracle.nvfp4_quantize(oracle.bf16_to_f32(host[sample]), amax=amax)
    assert to_np(gd)[0] == rg
    assert first_mismatch(to_np(c)[0][sample], rc) is None
    assert first_mismatch(to_np(s)[0][sample], rs) is None


def test_requant_stream_w_full_size_sampled_experts():
    E, rows, cols = 384, 2048, 4096
    g = inputs.device_generator(4, 1, DEV)
    w = inputs.device_normal((E * rows, cols), 0.02, g, DEV).view(torch.int16)
    c, s, gd = nvfp4_quantize(w, E, rows, cols)
    cn, sn, gn = to_np(c), to_np(s), to_np(gd)
    for e in [0, 191, 383]:
        host = to_np(w[e * rows:(e + 1) * rows], np.uint16)
        x32 = oracle.bf16_to_f32(host)
        amax = np.abs(x32).max()
        pick = np.random.default_rng(e).choice(rows, 16, replace=False)
        rc, rs, rg = oracle.nvfp4_quantize(x32[pick], amax=amax)
        assert gn[e] == rg
        assert first_mismatch(cn[e][pick], rc) is None and first_mismatch(sn[e][pick], rs) is None


@pytest.mark.parametrize("shape", [(4, 128), (37, 256), (256, 512)])
def test_hadamard_codec(shape):
    rows, cols = shape
    rng = np.random.default_rng(rows)
    x = rng.standard_t(3, (rows, cols)).astype(np.float32)
    x[rng.random(x.shape) < 0.003] *= 50
    xb = inputs.to_bf16_bits(x)
    codes = empty_u8(rows, cols // 2)
    sf = empty_u8(rows, cols // 16)
    gd = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_HADAMARD_QUANT))
    moe4.hadamard_quant(to_dev(xb), rows, cols, codes, sf, gd, moe4.FOUR_OVER_SIX, ws)
    out = torch.empty((rows, cols), dtype=torch.int16, device=DEV)
    moe4.hadamard_dequant(codes, sf, gd, rows, cols, out)
    torch.cuda.synchronize()
    rc, rs, rg = oracle.hadamard_quant(oracle.bf16_to_f32(xb))
    assert first_mismatch(to_np(codes), rc) is None
    assert first_mismatch(to_np(sf), rs) is None
    assert to_np(gd)[0] == rg
    ref = oracle.hadamard_dequant(rc, rs, rg)
    assert first_mismatch(to_np(out, np.uint16), ref) is None


def _mx_codec(x_dev, rows, cols):
    q = empty_u8(rows, cols)
    e8 = empty_u8(rows, cols // 32)
    moe4.hadamard_quant(x_dev, rows, cols, q, e8, None, moe4.MXFP8)
    out = torch.empty((rows, cols), dtype=torch.int16, device=DEV)
    moe4.hadamard_dequant(q, e8, None, rows, cols, out, moe4.MXFP8)
    torch.cuda.synchronize()
    return q, e8, out


@pytest.mark.parametrize("shape", [(4, 128), (37, 256), (256, 512), (3, 4096)])
def test_hadamard_mx_codec(shape):
    """The 8.25-bit variant (rotation, then MXFP8 per 32) against the oracle, bit for bit; row 0
    is all zero and row 1 tiny (scales in the subnormal range)."""
    rows, cols = shape
    rng = np.random.default_rng(100 + rows)
    x = rng.standard_t(3, (rows, cols)).astype(np.float32)
    x[rng.random(x.shape) < 0.003] *= 50
    x[0] = 0.0
    x[1] *= 1e-36
    xb = inputs.to_bf16_bits(x)
    q, e8, out = _mx_codec(to_dev(xb), rows, cols)
    rq, re = oracle.hadamard_quant_mx(oracle.bf16_to_f32(xb))
    assert first_mismatch(to_np(q), rq) is None
    assert first_mismatch(to_np(e8), re) is None
    assert first_mismatch(to_np(out, np.uint16), oracle.hadamard_dequant_mx(rq, re)) is None


def test_hadamard_mx_dequant_arbitrary_codes():
    """Decoder alone on codes the encoder would not emit: every non-NaN E4M3 byte, scales from
    2^-127 (E8M0 byte 0) up to 2^13."""
    rows, cols = 64, 1024
    rng = np.random.default_rng(7)
    finite = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)
    q = rng.choice(finite, (rows, cols))
    e8 = rng.integers(0, 141, (rows, cols // 32)).astype(np.uint8)
    e8[0] = 0
    out = torch.empty((rows, cols), dtype=torch.int16, device=DEV)
    moe4.hadamard_dequant(to_dev(q), to_dev(e8), None, rows, cols, out, moe4.MXFP8)
    torch.cuda.synchronize()
    assert first_mismatch(to_np(out, np.uint16), oracle.hadamard_dequant_mx(q, e8)) is None


def _codec_full_size_input():
    rows, cols = 131072, 4096  # the return-path tensor of 16384 tokens x top-8 at d = 4096
    g = inputs.device_generator(5, 0, DEV)
    return rows, cols, inputs.device_student_t((rows, cols), g, DEV).view(torch.int16)


def test_hadamard_codecs_full_size_sampled_rows():
    rows, cols, xb = _codec_full_size_input()
    host = to_np(xb, np.uint16)
    sample = np.concatenate([np.random.default_rng(5).choice(rows, 48, replace=False), [0, rows - 1]])
    xs = oracle.bf16_to_f32(host[sample])

    q, e8, out = _mx_codec(xb, rows, cols)
    rq, re = oracle.hadamard_quant_mx(xs)
    assert first_mismatch(to_np(q[sample]), rq) is None
    assert first_mismatch(to_np(e8[sample]), re) is None
    assert first_mismatch(to_np(out[sample], np.uint16), oracle.hadamard_dequant_mx(rq, re)) is None
    del q, e8

    codes = empty_u8(rows, cols // 2)
    sf = empty_u8(rows, cols // 16)
    gd = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_HADAMARD_QUANT))
    moe4.hadamard_quant(xb, rows, cols, codes, sf, gd, moe4.FOUR_OVER_SIX, ws)
    moe4.hadamard_dequant(codes, sf, gd, rows, cols, out)
    torch.cuda.synchronize()
    amax = 0.0
    for r0 in range(0, rows, 8192):  # the rotated tensor's amax sets the per-tensor scale
        amax = max(amax, float(np.abs(oracle.hadamard_rotate(oracle.bf16_to_f32(host[r0:r0 + 8192]))).max()))
    rc, rs, rg = oracle.nvfp4_quantize(oracle.hadamard_rotate(xs), amax=amax)
    assert to_np(gd)[0] == rg
    assert first_mismatch(to_np(codes[sample]), rc) is None
    assert first_mismatch(to_np(sf[sample]), rs) is None
    assert first_mismatch(to_np(out[sample], np.uint16), oracle.hadamard_dequant(rc, rs, rg)) is None


def test_hadamard_mx_codec_empty_and_bad_flags():
    q = empty_u8(1, 128)
    e8 = empty_u8(1, 4)
    moe4.hadamard_quant(None, 0, 128, q, e8, None, moe4.MXFP8)
    x = torch.zeros((1, 128), dtype=torch.int16, device=DEV)
    with pytest.raises(RuntimeError):
        moe4.hadamard_quant(x, 1, 128, q, e8, None, moe4.MXFP8 | moe4.FOUR_OVER_SIX)
    with pytest.raises(RuntimeError):
        moe4.hadamard_quant(x, 1, 96, q, e8, None, moe4.MXFP8)


def _device_patterns(start, count):
    bits = torch.arange(start, start + count, dtype=torch.int64, device=DEV)
    return (bits - (bits >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32).view(torch.float32)


@pytest.mark.parametrize("sign", [0, 1])
def test_device_e2m1_conversion_exhaustive_binades(sign):
    lo = (sign << 31) | (123 << 23)
    step = 1 << 24
    for start in range(lo, lo + (8 << 23), step):
        v = _device_patterns(start, step)
        out = torch.empty(step, dtype=torch.uint8, device=DEV)
        moe4.moe4_convert(0, v, step, out)
        torch.cuda.synchronize()
        assert first_mismatch(to_np(out), oracle.e2m1_range(start, step)) is None


def test_device_e4m3_conversion_exhaustive_binades():
    step = 1 << 24
    for sign in (0, 1):
        lo, hi = (sign << 31) | (115 << 23), (sign << 31) | (136 << 23)
        for start in range(lo, hi, step):
            n = min(step, hi - start)
            v = _device_patterns(start, n)
            out = torch.empty(n, dtype=torch.uint8, device=DEV)
            moe4.moe4_convert(1, v, n, out)
            torch.cuda.synchronize()
            assert first_mismatch(to_np(out), oracle.e4m3_range(start, n)) is None


def test_device_conversions_strided_all_patterns():
    bits = np.arange(0, 1 << 32, 4099, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    v = v[: v.size // 4 * 4]
    vd = to_dev(v)
    for kind, ref in [(0, oracle.e2m1_rne_sat(v)), (1, oracle.e4m3_rne_sat(v))]:
        out = torch.empty(v.size, dtype=torch.uint8, device=DEV)
        moe4.moe4_convert(kind, vd, v.size, out)
        torch.cuda.synchronize()
        assert first_mismatch(to_np(out), ref) is None, kind
    out = torch.empty(v.size, dtype=torch.int16, device=DEV)
    moe4.moe4_convert(2, vd, v.size, out)
    torch.cuda.synchronize()
    assert first_mismatch(to_np(out, np.uint16), oracle.f32_to_bf16(v)) is None


def test_device_stochastic_rounding_and_words():
    rng = np.random.default_rng(9)
    n = 1 << 20
    v = (rng.standard_normal(n) * np.exp2(rng.integers(-14, 8, n))).astype(np.float32)
    v = np.clip(v, -448, 448).astype(np.float32)
    # edges of the four-at-a-time fast path: signed zeros, 2^-6 and its neighbours, 448, values
    # just under the top of a binade (carry into the exponent); the first groups of four are pure
    # edge cases, later ones mix one tiny value into normal ones
    edges = np.array([0.0, -0.0, 2.0 ** -6, -2.0 ** -6, np.nextafter(np.float32(2.0 ** -6), np.float32(0)),
                      -np.nextafter(np.float32(2.0 ** -6), np.float32(0)), 448.0, -448.0, 447.9, 415.9,
                      np.nextafter(np.float32(1.0), np.float32(0)), 1.0, 1e-30, -3e-3, 2.0 ** -9, 0.0],
                     np.float32)
    v[:edges.size] = edges
    v[1024:1024 + 4 * 64:4] = edges[np.arange(64) % edges.size]
    out = torch.empty(n, dtype=torch.uint8, device=DEV)
    moe4.moe4_convert(3, to_dev(v), n, out)
    words = torch.empty(n, dtype=torch.int16, device=DEV)
    moe4.moe4_sr_words(0x0123456789ABCDEF, 5, 1 << 33, n, words)
    torch.cuda.synchronize()
    ref_words0 = oracle.sr_words(0, 0, 0, n)
    assert first_mismatch(to_np(out), oracle.e4m3_sr(v, ref_words0)) is None
    assert first_mismatch(to_np(words, np.uint16), oracle.sr_words(0x0123456789ABCDEF, 5, 1 << 33, n)) is None


def test_full_tensor_parity_small_moe_operands():
    """Every block of the small-MoE GEMM operands: activations [8704, 2048] Student-t(3) and
    8 experts' weights [8, 2048, 2048] N(0, 0.02)."""
    rng = np.random.default_rng(13)
    a = inputs.to_bf16_bits((rng.standard_t(3, (8704, 2048)) / np.sqrt(3)).astype(np.float32))
    b = inputs.to_bf16_bits((rng.standard_normal((8 * 2048, 2048)) * 0.02).astype(np.float32))
    _check_quant(a, 1, 8704, 2048)
    _check_quant(b, 8, 2048, 2048)


@pytest.mark.parametrize("given,mma,ld", [(False, False, 256), (True, True, 256), (False, True, 260)])
def test_quantize_f32_equals_quantize_of_bf16_copy(given, mma, ld):
    """nvfp4_quantize_f32 rounds each binary32 value to bf16 as it reads it: its outputs equal the
    oracle's quantisation of the oracle's bf16 rounding of the same values (ties to even included:
    some values sit exactly halfway between two bf16 numbers), with or without a given amax, in
    both scale layouts, with padded rows."""
    nmat, rows, cols = 3, 128, 256
    rng = np.random.default_rng(61)
    x = (rng.standard_normal((nmat, rows, cols)) * np.array([0.02, 1.0, 30.0])[:, None, None]).astype(np.float32)
    bits = x.view(np.uint32)
    tie = rng.random(x.shape) < 0.05            # force the 16 dropped bits to exactly one half
    bits[tie] = (bits[tie] & 0xFFFF0000) | 0x8000
    xb = oracle.f32_to_bf16(x)                    # the bf16 copy, nearest-even
    amax = np.abs(oracle.bf16_to_f32(xb)).reshape(nmat, -1).max(axis=1).astype(np.float32)
    xpad = np.zeros((nmat, rows, ld), np.float32)
    xpad[:, :, :cols] = x
    c, s = empty_u8(nmat, rows, cols // 2), empty_u8(nmat, rows, cols // 16)
    g = torch.empty(nmat, dtype=torch.float32, device=DEV)
    flags = moe4.FOUR_OVER_SIX | (moe4.AMAX_GIVEN if given else 0) | (moe4.SF_MMA_LAYOUT if mma else 0)
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_NVFP4_QUANTIZE, nmat))
    moe4.nvfp4_quantize_f32(to_dev(xpad), nmat, rows, cols, ld, c, s, g, to_dev(amax) if given else None, flags, ws)
    torch.cuda.synchronize()
    rc, rs, rg = oracle.nvfp4_quantize(oracle.bf16_to_f32(xb))
    assert first_mismatch(to_np(g), rg) is None
    assert first_mismatch(to_np(c), rc) is None
    s_np = to_np(s)
    if mma:
        s2 = empty_u8(nmat, rows, cols // 16)
        moe4.moe4_sf_to_mma_layout(to_dev(rs), nmat, rows, cols // 16, s2)
        torch.cuda.synchronize()
        assert np.array_equal(s_np, to_np(s2))
    else:
        assert first_mismatch(s_np, rs) is None


@pytest.mark.parametrize("mx", [False, True])
def test_hadamard_codecs_on_subnormal_rows(mx):
    """Rows at the bottom of the bf16 range: every value subnormal (so the butterflies' sums and
    differences are subnormal too), subnormal values beside one normal value, and normal values
    whose differences cancel into the subnormal range; both return-path codecs against the
    oracle, bit for bit, codes and decoded rows."""
    rows, cols = 8, 256
    rng = np.random.default_rng(41)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x[0:3] *= 1e-39                                  # all subnormal
    x[3] *= 1e-39
    x[3, 7] = 1.0                                    # one normal value among subnormals
    x[4] = np.float32(2.0 ** -125) * np.sign(x[4])   # equal magnitudes at the normal edge: exact cancellations
    x[5] = (np.float32(2.0 ** -126) * (1 + (rng.integers(0, 4, cols) / 8.0)) * np.sign(x[5])).astype(np.float32)
    xb = inputs.to_bf16_bits(x)
    if mx:
        q, e8, out = _mx_codec(to_dev(xb), rows, cols)
        rq, re = oracle.hadamard_quant_mx(oracle.bf16_to_f32(xb))
        assert first_mismatch(to_np(q), rq) is None
        assert first_mismatch(to_np(e8), re) is None
        assert first_mismatch(to_np(out, np.uint16), oracle.hadamard_dequant_mx(rq, re)) is None
    else:
        codes, sf = empty_u8(rows, cols // 2), empty_u8(rows, cols // 16)
        gd = torch.empty(1, dtype=torch.float32, device=DEV)
        ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_HADAMARD_QUANT))
        moe4.hadamard_quant(to_dev(xb), rows, cols, codes, sf, gd, moe4.FOUR_OVER_SIX, ws)
        out = torch.empty((rows, cols), dtype=torch.int16, device=DEV)
        moe4.hadamard_dequant(codes, sf, gd, rows, cols, out)
        torch.cuda.synchronize()
        rc, rs, rg = oracle.hadamard_quant(oracle.bf16_to_f32(xb))
        assert first_mismatch(to_np(codes), rc) is None
        assert first_mismatch(to_np(sf), rs) is None
        assert np.array_equal(to_np(gd), np.atleast_1d(rg))
        assert first_mismatch(to_np(out, np.uint16), oracle.hadamard_dequant(rc, rs, rg)) is None


@pytest.mark.parametrize("fos", [True, False])
def test_quantize_subnormal_inputs(fos):
    """NVFP4 of tensors at the bottom of the bf16 range, against the oracle bit for bit: a whole
    matrix of random subnormal values (the per-tensor scale then lifts them into range), and a
    normal matrix whose 16-column blocks 3 and 10 hold only subnormal values (their block scale
    underflows to zero), except one normal value in block 10 of row 5."""
    rng = np.random.default_rng(43)
    a = (rng.standard_normal((64, 256)) * 1e-39).astype(np.float32)
    b = rng.standard_t(3, (64, 256)).astype(np.float32)
    b[:, 48:64] *= 1e-39
    b[:, 160:176] *= 1e-39
    b[5, 160] = 3.0
    xb = inputs.to_bf16_bits(np.stack([a, b]))
    _check_quant(xb, 2, 64, 256, fos=fos)


@pytest.mark.parametrize("f32,mma", [(False, False), (False, True), (True, False), (True, True)])
def test_quantize_strided_rows_several_blocks_per_thread(f32, mma):
    """Padded rows (ld > cols) on a stack large enough that every thread of the quantiser's grid
    takes several blocks, two per loop iteration, pairs crossing matrix boundaries: codes, scales
    (canonical or tile layout) and g_dec against the oracle, bit for bit."""
    nmat, rows, cols, ld = 5, 2048, 2048, 2080
    rng = np.random.default_rng(71 + 2 * f32 + mma)
    x = rng.standard_t(3, (nmat, rows, cols)).astype(np.float32)
    x *= np.exp2(rng.integers(-6, 6, (nmat, 1, 1))).astype(np.float32)
    xb = oracle.f32_to_bf16(x)
    pad = np.zeros((nmat, rows, ld), np.float32 if f32 else np.uint16)
    pad[:, :, :cols] = x if f32 else xb
    c, s = empty_u8(nmat, rows, cols // 2), empty_u8(nmat, rows, cols // 16)
    g = torch.empty(nmat, dtype=torch.float32, device=DEV)
    flags = moe4.FOUR_OVER_SIX | (moe4.SF_MMA_LAYOUT if mma else 0)
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_NVFP4_QUANTIZE, nmat))
    quant = moe4.nvfp4_quantize_f32 if f32 else moe4.nvfp4_quantize
    quant(to_dev(pad), nmat, rows, cols, ld, c, s, g, None, flags, ws)
    torch.cuda.synchronize()
    rc, rs, rg = oracle.nvfp4_quantize(oracle.bf16_to_f32(xb))
    assert first_mismatch(to_np(g), rg) is None
    assert first_mismatch(to_np(c), rc) is None
    if mma:
        s2 = empty_u8(nmat, rows, cols // 16)
        moe4.moe4_sf_to_mma_layout(to_dev(rs), nmat, rows, cols // 16, s2)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(s), to_np(s2))
    else:
        assert first_mismatch(to_np(s), rs) is None
