"""Pins of the oracle's Hadamard return-path codec ("4-bit computation from the start of Inkling 2
Small's pretraining", lhc.media, communication paragraph: a Hadamard transform spreads out
extreme values before the return path is quantised).

Pins: H H = 128 I in integers for the Sylvester matrix; the butterfly of every unit vector is
the matching Hadamard column times the binary32 constant; the constant is the nearest binary32
to 1/sqrt(128); the transform against an explicit float64 matrix product; self-inverse to a few
ulp; a one-hot spike becomes a flat row (amax drops by sqrt(128)); and the codec is the rotation
followed by NVFP4 (and the inverse) with a bounded round-trip error.
"""
from fractions import Fraction

import numpy as np


def _sylvester(n):
    H = np.array([[1]], np.int64)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def test_sylvester_orthogonality():
    H = _sylvester(128)
    assert np.array_equal(H @ H, 128 * np.eye(128, dtype=np.int64))


def test_scale_constant_is_nearest_binary32(orc):
    c = orc.hadamard_scale()
    assert np.array([c], np.float32).view(np.uint32)[0] == 0x3DB504F3
    lo = Fraction(float(np.nextafter(c, np.float32(0))))
    hi = Fraction(float(np.nextafter(c, np.float32(1))))
    fc = Fraction(float(c))
    m_lo, m_hi = (lo + fc) / 2, (fc + hi) / 2
    assert m_lo * m_lo < Fraction(1, 128) < m_hi * m_hi


def test_unit_vectors_give_hadamard_columns(orc):
    H = _sylvester(128)
    c = orc.hadamard_scale()
    for i in range(128):
        e = np.zeros(128, np.float32)
        e[i] = 1.0
        got = orc.fwht128(e)
        assert np.array_equal(got, (H[:, i] * c).astype(np.float32)), i


def test_against_matrix_product(orc):
    H = _sylvester(128).astype(np.float64)
    rng = np.random.default_rng(0)
    x = rng.standard_t(3, (64, 128)).astype(np.float32)
    got = orc.hadamard_rotate(x).astype(np.float64)
    want = (x.astype(np.float64) @ H.T) * float(orc.hadamard_scale())
    bound = 8 * 2.0 ** -24 * (np.abs(x).astype(np.float64) @ np.abs(H).T) * float(orc.hadamard_scale())
    assert np.all(np.abs(got - want) <= bound + 1e-30)


def test_self_inverse(orc):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((32, 256)).astype(np.float32)
    back = orc.hadamard_rotate(orc.hadamard_rotate(x))
    assert np.max(np.abs(back - x) / np.abs(x).max(axis=1, keepdims=True)) < 1e-6


def test_spike_becomes_flat(orc):
    x = np.zeros((1, 128), np.float32)
    x[0, 37] = 100.0
    r = orc.hadamard_rotate(x)
    assert np.allclose(np.abs(r), 100.0 * float(orc.hadamard_scale()))
    assert np.isclose(np.abs(x).max() / np.abs(r).max(), np.sqrt(128), rtol=1e-6)


def test_codec_definition_and_round_trip(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((256, 512)).astype(np.float32)
    spikes = rng.random(x.shape) < 0.002
    x = np.where(spikes, x * 200, x).astype(np.float32)
    codes, sf, g = orc.hadamard_quant(x)
    c2, s2, g2 = orc.nvfp4_quantize(orc.hadamard_rotate(x))
    assert np.array_equal(codes, c2) and np.array_equal(sf, s2) and g == g2
    back = orc.bf16_to_f32(orc.hadamard_dequant(codes, sf, g))
    want = orc.bf16_to_f32(orc.f32_to_bf16(orc.hadamard_rotate(orc.nvfp4_dequantize(codes, sf, g))))
    assert np.array_equal(back, want)
    # the round trip stays within NVFP4's error on these rows (it is not smaller: with 16-value
    # blocks a spike only coarsens its own block, and the rotation spreads it over eight)
    err_h = np.linalg.norm(back - x) / np.linalg.norm(x)
    assert err_h < 0.1


def test_mx_codec_is_8_25_bits_per_value(orc):
    # the pages' return-path payload: sixteen -> 8.25 bits per value
    x = np.random.default_rng(3).standard_normal((64, 512)).astype(np.float32)
    q, e8 = orc.hadamard_quant_mx(x)
    assert (q.nbytes + e8.nbytes) * 8 / x.size == 8.25
    assert 16 / ((q.nbytes + e8.nbytes) * 8 / x.size) == 16 / 8.25


def test_mx_codec_definition_and_round_trip(orc):
    rng = np.random.default_rng(4)
    x = rng.standard_t(3, (128, 256)).astype(np.float32)
    x[rng.random(x.shape) < 0.003] *= 100
    q, e8 = orc.hadamard_quant_mx(x)
    q2, e82 = orc.mxfp8_quantize_rows(orc.hadamard_rotate(x), sr=False)
    assert np.array_equal(q, q2) and np.array_equal(e8, e82)
    back = orc.bf16_to_f32(orc.hadamard_dequant_mx(q, e8))
    want = orc.bf16_to_f32(orc.f32_to_bf16(orc.hadamard_rotate(orc.mxfp8_dequantize(q, e8))))
    assert np.array_equal(back, want)
    # 8-bit elements: the round trip is far tighter than the 4-bit codec's
    err_mx = np.linalg.norm(back - x) / np.linalg.norm(x)
    cq, sq, gq = orc.hadamard_quant(x)
    err_fp4 = np.linalg.norm(orc.bf16_to_f32(orc.hadamard_dequant(cq, sq, gq)) - x) / np.linalg.norm(x)
    assert err_mx < 0.05 and err_mx < err_fp4 / 2


def test_mx_codec_spreads_a_spike(orc):
    # a lone spike forces a large scale on its 32-block without the rotation; rotated, every value
    # of its 128-chunk is the same size and the chunk's other values keep their precision
    x = np.full((1, 128), 0.01, np.float32)
    x[0, 5] = 1000.0
    q, e8 = orc.hadamard_quant_mx(x)
    assert len(set(e8[0].tolist())) == 1          # four equal block scales after rotation
    qp, e8p = orc.mxfp8_quantize_rows(x, sr=False)
    assert e8p[0, 0] > e8p[0, 1]                 # without it, the spike's block scale stands out
