"""Pins of the oracle's number formats against things other than the oracle itself.

- the E2M1 code set fixed for NVFP4 (tests/golden/e2m1_code_set.txt);
- E2M1 nearest-even rounding recomputed by a different method (numpy's half-to-even round of
  the quotient by the binade spacing), over every binary32 pattern in [2^-4, 2^4) of both signs
  plus a strided sample of all 2^32 patterns;
- E4M3 nearest-even rounding against torch's float8_e4m3fn cast (a library routine) over every
  binary32 pattern in [2^-12, 2^9) and the saturation rule above it;
- bf16 nearest-even against torch's bfloat16 cast;
- bits per value: 4.5 for NVFP4 (four-bit values plus one 8-bit scale per sixteen, "4-bit
  computation from the start of Inkling 2 Small's pretraining", fewer-bits paragraph), 16/4.5 =
  3.6x fewer than BF16 ("Thinking Machines: Nvidia FP4 Up to 6x Faster, Runs Gain 8%", "What
  Thinking Machines Changed"), and 8.25 for 32-blocks of 8-bit values with an 8-bit scale (the
  return-path figure of the lhc.media communication paragraph).
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_code_set():
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_code_set.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            table[int(c)] = float(v)
    return table


def test_e2m1_code_set_matches_pages(orc):
    table = _load_code_set()
    assert sorted(table) == list(range(16))
    vals = orc.e2m1_value(np.arange(16, dtype=np.uint8))
    for c in range(16):
        assert vals[c] == table[c]
        assert np.signbit(vals[c]) == (c >= 8)


def _e2m1_by_np_round(v: np.ndarray) -> np.ndarray:
    """Independent E2M1 rounding: for |v| < 1 the spacing is 0.5, in [2^E, 2^(E+1)) (E = 0, 1, 2) it
    is 2^(E-1); round the quotient half-to-even with numpy, saturate at 6, and read the code off
    the value."""
    a = np.abs(v.astype(np.float64))
    spacing = np.where(a < 1.0, 0.5, np.exp2(np.floor(np.log2(np.maximum(a, 1.0))) - 1.0))
    spacing = np.where(a >= 4.0, 2.0, spacing)
    mag = np.round(a / spacing) * spacing
    mag = np.minimum(mag, 6.0)
    value_to_code = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
    lut_keys = np.array(sorted(value_to_code))
    idx = np.searchsorted(lut_keys, mag)
    assert np.all(lut_keys[idx] == mag)
    codes = np.array([value_to_code[k] for k in lut_keys], np.uint8)[idx]
    return codes | (np.signbit(v).astype(np.uint8) << 3)


def test_e2m1_ties_and_saturation(orc):
    cases = {0.25: 0, 0.2500001: 1, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             5.0001: 7, 6.0: 7, 7.0: 7, 1e30: 7, 0.0: 0}
    for v, code in cases.items():
        assert orc.e2m1_rne_sat([v])[0] == code, v
        assert orc.e2m1_rne_sat([-v])[0] == code | 8, -v
    assert orc.e2m1_rne_sat([-1e-7])[0] == 0x8  # small negatives keep their sign (-0)


@pytest.mark.parametrize("sign", [0, 1])
def test_e2m1_exhaustive_binades(orc, sign):
    lo = (sign << 31) | (123 << 23)   # 2^-4
    hi = (sign << 31) | (131 << 23)   # 2^4
    step = 1 << 23
    for start in range(lo, hi, step):
        bits = np.arange(start, start + step, dtype=np.uint64).astype(np.uint32)
        got = orc.e2m1_range(start, step)
        want = _e2m1_by_np_round(bits.view(np.float32))
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, hex(int(bits[bad[0]]))


def test_e2m1_strided_all_patterns(orc):
    bits = np.arange(0, 1 << 32, 65537, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    finite = np.isfinite(v)
    got = orc.e2m1_rne_sat(v[finite])
    want = _e2m1_by_np_round(v[finite])
    assert np.array_equal(got, want)


def test_e4m3_against_torch_exhaustive(orc):
    lo = 115 << 23    # 2^-12
    hi = 136 << 23    # 2^9 (=512), then compare only below 464 where torch does not produce NaN
    step = 1 << 23
    for start in range(lo, hi, step):
        bits = np.arange(start, start + step, dtype=np.uint64).astype(np.uint32)
        v = bits.view(np.float32)
        keep = v < 464.0
        got = orc.e4m3_range(start, step)[keep]
        want = torch.from_numpy(v[keep]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, hex(int(bits[keep][bad[0]]))
    # below 2^-12 everything is +0; from 448 up everything saturates to 448 (0x7E)
    assert np.all(orc.e4m3_rne_sat(np.array([2.0 ** -11, 1e-30, 0.0], np.float32)) == 0)
    assert orc.e4m3_rne_sat([2.0 ** -10 * 1.0000001])[0] == 1
    big = np.array([448.0, 460.0, 464.0, 470.0, 480.0, 1e6, 3e38], np.float32)
    assert np.all(orc.e4m3_rne_sat(big) == 0x7E)
    assert np.all(orc.e4m3_rne_sat(-big) == 0xFE)


def test_e4m3_values(orc):
    v = orc.e4m3_value(np.arange(256, dtype=np.uint8))
    assert v[0x7E] == 448.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9 and v[0x38] == 1.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)  # codes are in value order
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    fin = ~np.isnan(ref)
    assert np.array_equal(v[fin], ref[fin])


def test_e8m0_values(orc):
    v = orc.e8m0_value(np.array([0, 1, 126, 127, 128, 254], np.uint8))
    assert list(v) == [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 127]


def test_bf16_against_torch(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 3.3e38)]
    v = np.concatenate([v, np.float32([1.00390625, 1.01171875, -0.0, 0.0, 65504.0])])
    got = orc.f32_to_bf16(v)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    back = orc.bf16_to_f32(got)
    assert np.array_equal(back, torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_bits_per_value():
    cols = 4096
    nvfp4_bits = (cols // 2 + cols // 16) * 8 / cols
    assert nvfp4_bits == 4.5
    assert round(16 / nvfp4_bits, 1) == 3.6
    mxfp8_bits = (cols + cols // 32) * 8 / cols
    assert mxfp8_bits == 8.25
