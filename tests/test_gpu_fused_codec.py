"""GPU parity of the down-projection GEMM with the return-path codec fused into its final stage
("4-bit computation from the start of Inkling 2 Small's pretraining": kernels paragraph for the
fusion, communication paragraph for the Hadamard transform and the 8.25 bits per value).

1. Byte for byte against the two unfused calls on the device: grouped_expert_gemm_nvfp4 with a
   bf16 product, then hadamard_quant with MOE4_MXFP8.  Each of those has its own parity tests
   against the oracle (the GEMM within its accumulation bound, the codec bit for bit).
2. End to end against the oracle: its float64 GEMM of its own NVFP4 operands, rounded to bf16,
   through its 8.25-bit codec.  Both sides are decoded by the oracle; per 128-value chunk the
   difference is bounded by the bf16 product difference plus each side's MXFP8 rounding error
   (at most 2^-4 of a normal-range value, or half the subnormal step 2^(e-10), per element; the
   rotations preserve the L2 norm).  As a structural check most code bytes must agree exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import inputs, moe4
from gpu_helpers import DEV, empty_u8, nvfp4_quantize, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    moe4.load()


def _offs(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _run_both(h_bits, w_bits, offs, E, N, K):
    """h_bits [R, K], w_bits [E*N, K]: device int16 tensors of bf16 bits."""
    R = int(offs[-1])
    ac, asf, ag = nvfp4_quantize(h_bits, 1, R, K)
    bc, bsf, bg = nvfp4_quantize(w_bits, E, N, K)
    offs_d = to_dev(offs)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(0, R, E, N, K))
    q, e8 = empty_u8(R, N), empty_u8(R, N // 32)
    moe4.grouped_expert_gemm_nvfp4_hadamard_mx(ac, asf, ag, bc, bsf, bg, offs_d, E, R, N, K, q, e8, 0, ws)
    y = torch.empty((R, N), dtype=torch.int16, device=DEV)
    moe4.grouped_expert_gemm_nvfp4(ac, asf, ag, bc, bsf, bg, offs_d, E, R, N, K, y, moe4.OUT_BF16, ws)
    q2, e82 = empty_u8(R, N), empty_u8(R, N // 32)
    moe4.hadamard_quant(y, R, N, q2, e82, None, moe4.MXFP8)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    return q, e8, q2, e82


def test_fused_equals_unfused_small_groups():
    rng = np.random.default_rng(41)
    sizes = [256, 128, 0, 384, 128, 256, 0, 128]
    E, N, K = len(sizes), 512, 512
    offs = _offs(sizes)
    R = int(offs[-1])
    h = inputs.to_bf16_bits((rng.standard_t(3, (R, K)) / np.sqrt(3)).astype(np.float32))
    w = inputs.to_bf16_bits((rng.standard_normal((E * N, K)) * 0.02).astype(np.float32))
    q, e8, q2, e82 = _run_both(to_dev(h), to_dev(w), offs, E, N, K)
    assert torch.equal(q, q2) and torch.equal(e8, e82)


def test_fused_equals_unfused_full_size():
    """The down projection of the 384-expert layer: 160512 padded rows, d_model 4096, width 2048."""
    rng = np.random.default_rng(0)
    counts = rng.multinomial(16384 * 8, rng.dirichlet(np.ones(384) * 0.5))
    offs = _offs((counts + 127) // 128 * 128)
    E, N, K = 384, 4096, 2048
    R = int(offs[-1])
    h = inputs.device_normal((R, K), 1.0, inputs.device_generator(8, 0, DEV), DEV).view(torch.int16)
    w = inputs.device_normal((E * N, K), 0.02, inputs.device_generator(8, 1, DEV), DEV).view(torch.int16)
    q, e8, q2, e82 = _run_both(h, w, offs, E, N, K)
    assert torch.equal(q, q2) and torch.equal(e8, e82)


def test_fused_against_oracle_end_to_end():
    rng = np.random.default_rng(43)
    sizes = [128, 256, 0, 128]
    E, N, K = len(sizes), 512, 256
    offs = _offs(sizes)
    R = int(offs[-1])
    h = inputs.to_bf16_bits((rng.standard_t(3, (R, K)) / np.sqrt(3)).astype(np.float32))
    w = inputs.to_bf16_bits((rng.standard_normal((E * N, K)) * 0.02).astype(np.float32))
    q, e8, _, _ = _run_both(to_dev(h), to_dev(w), offs, E, N, K)
    # oracle: quantise its own operands, float64 GEMM, bf16, 8.25-bit codec
    rac, ras, rag = oracle.nvfp4_quantize(oracle.bf16_to_f32(h))
    rbc, rbs, rbg = oracle.nvfp4_quantize(oracle.bf16_to_f32(w).reshape(E, N, K))
    D, S = oracle.grouped_gemm_m(oracle.nvfp4_dequantize(rac, ras, rag), oracle.nvfp4_dequantize(rbc, rbs, rbg), offs)
    yr = oracle.f32_to_bf16(D.astype(np.float32))
    rq, re8 = oracle.hadamard_quant_mx(oracle.bf16_to_f32(yr))
    got = oracle.bf16_to_f32(oracle.hadamard_dequant_mx(to_np(q), to_np(e8))).astype(np.float64)
    ref = oracle.bf16_to_f32(oracle.hadamard_dequant_mx(rq, re8)).astype(np.float64)
    # per-chunk bound
    delta = 2.0 ** -16 * S * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(D)   # |bf16 product difference|
    yabs = np.abs(oracle.bf16_to_f32(yr).astype(np.float64))
    chunks = lambda a: a.reshape(R, N // 128, 128)
    d_norm = np.linalg.norm(chunks(delta), axis=2)
    y_norm = np.linalg.norm(chunks(yabs), axis=2)
    # a rotated value is at most the chunk's L2 norm, so each block's 2^e < 2 * norm / 448
    sub_floor = np.sqrt(128.0) * 2 * (y_norm + d_norm) / (448.0 * 1024)
    # + both decoders' bf16 rounding (2^-9 relative) and the binary32 rotations (far below 1e-6)
    bound = (d_norm + 2.0 ** -4 * (2 * y_norm + d_norm) + 2 * sub_floor
             + 2.0 ** -8 * (y_norm + d_norm) * (1 + 2.0 ** -4) + 1e-6 * y_norm + 1e-30)
    err = np.linalg.norm(chunks(got - ref), axis=2)
    assert np.all(err <= bound), "worst chunk err/bound %.3f" % float(np.max(err / bound))
    assert np.mean(to_np(q) == rq) >= 0.9 and np.mean(to_np(e8) == re8) >= 0.9


def _nvfp4_codec_case(h, w, offs, E, N, K):
    """The down projection with the rotated amax from its last stage, then the NVFP4 return-path
    encoder taking that amax; beside it the plain bf16 GEMM and the encoder's own amax pass."""
    R = int(offs[-1])
    ac, asf, ag = nvfp4_quantize(h, 1, R, K)
    bc, bsf, bg = nvfp4_quantize(w, E, N, K)
    offs_d = to_dev(offs)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(0, R, E, N, K))
    y1 = torch.empty((R, N), dtype=torch.int16, device=DEV)
    amax = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
    moe4.grouped_expert_gemm_nvfp4_hadamard_amax(ac, asf, ag, bc, bsf, bg, offs_d, E, R, N, K, y1, amax, 0, ws)
    c1, s1, g1 = empty_u8(R, N // 2), empty_u8(R, N // 16), torch.empty(1, dtype=torch.float32, device=DEV)
    moe4.hadamard_quant(y1, R, N, c1, s1, g1, moe4.FOUR_OVER_SIX | moe4.AMAX_GIVEN, amax)
    y2 = torch.empty((R, N), dtype=torch.int16, device=DEV)
    moe4.grouped_expert_gemm_nvfp4(ac, asf, ag, bc, bsf, bg, offs_d, E, R, N, K, y2, moe4.OUT_BF16, ws)
    c2, s2, g2 = empty_u8(R, N // 2), empty_u8(R, N // 16), torch.empty(1, dtype=torch.float32, device=DEV)
    hws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_HADAMARD_QUANT))
    moe4.hadamard_quant(y2, R, N, c2, s2, g2, moe4.FOUR_OVER_SIX, hws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    assert torch.equal(y1, y2)
    assert torch.equal(amax.view(torch.int32), hws[:4].view(torch.int32))
    assert torch.equal(c1, c2) and torch.equal(s1, s2) and torch.equal(g1, g2)
    return y1, amax, c1, s1, g1


def test_nvfp4_codec_amax_from_gemm_small_groups():
    """The NVFP4 return path with its amax taken in the GEMM's last stage equals the bf16 GEMM
    followed by the two-pass encoder, byte for byte, and both equal the oracle's encoder of the
    same bf16 product."""
    rng = np.random.default_rng(44)
    sizes = [256, 128, 0, 384, 128]
    E, N, K = len(sizes), 512, 512
    offs = _offs(sizes)
    h = inputs.to_bf16_bits((rng.standard_t(3, (int(offs[-1]), K)) / np.sqrt(3)).astype(np.float32))
    w = inputs.to_bf16_bits((rng.standard_normal((E * N, K)) * 0.02).astype(np.float32))
    y, amax, c, s, g = _nvfp4_codec_case(to_dev(h), to_dev(w), offs, E, N, K)
    rc, rs, rg = oracle.hadamard_quant(oracle.bf16_to_f32(to_np(y, np.uint16)))
    assert np.array_equal(to_np(c), rc) and np.array_equal(to_np(s), rs) and float(to_np(g)[0]) == float(rg)


def test_nvfp4_codec_amax_from_gemm_layer_shape():
    """At the layer step's down-projection shape (384 experts, 160512 padded rows, d_model 4096,
    width 2048): the same byte-for-byte equality, and sampled rows against the oracle: its
    rotation of the whole bf16 product gives the amax, then its NVFP4 quantiser encodes the
    sampled rotated rows with that amax ("4-bit computation from the start of Inkling 2 Small's
    pretraining", communication and kernels paragraphs)."""
    rng = np.random.default_rng(0)
    counts = rng.multinomial(16384 * 8, rng.dirichlet(np.ones(384) * 0.5))
    offs = _offs((counts + 127) // 128 * 128)
    E, N, K = 384, 4096, 2048
    R = int(offs[-1])
    h = inputs.device_student_t((R, K), inputs.device_generator(9, 0, DEV), DEV).view(torch.int16)
    w = inputs.device_normal((E * N, K), 0.02, inputs.device_generator(9, 1, DEV), DEV).view(torch.int16)
    y, amax, c, s, g = _nvfp4_codec_case(h, w, offs, E, N, K)
    del h, w
    rot = oracle.hadamard_rotate(oracle.bf16_to_f32(to_np(y, np.uint16)))
    ref_amax = np.float32(np.abs(rot).max())
    assert float(to_np(amax)[0]) == float(ref_amax)
    rows = np.unique(np.random.default_rng(3).choice(R, 64, replace=False))
    rc, rs, rg = oracle.nvfp4_quantize(rot[rows], amax=ref_amax)
    assert float(to_np(g)[0]) == float(rg)
    assert np.array_equal(to_np(c)[rows], rc) and np.array_equal(to_np(s)[rows], rs)


def _plan(T, E, k, seed):
    rng = np.random.default_rng(seed)
    lg = (rng.standard_normal((T, E)) + rng.standard_normal(E)).astype(np.float32)
    idx, w = oracle.route_topk(lg, k)
    offs, row_of = oracle.permute_plan(idx, E)
    return offs, row_of, w


@pytest.mark.parametrize("T,E,k,d", [(300, 16, 4, 256), (16384, 384, 8, 4096)])
def test_combine_from_encoded_return_path(T, E, k, d):
    """moe4_combine_hadamard (decode + combine in one pass) equals hadamard_dequant followed by
    moe4_combine byte for byte; the small case also equals the oracle's decode and combine."""
    offs, row_of, w = _plan(T, E, k, 50 + T)
    R = int(offs[-1])
    yb = inputs.device_student_t((R, d), inputs.device_generator(50, T, DEV), DEV).view(torch.int16)
    c, s = empty_u8(R, d // 2), empty_u8(R, d // 16)
    g = torch.empty(1, dtype=torch.float32, device=DEV)
    moe4.hadamard_quant(yb, R, d, c, s, g, moe4.FOUR_OVER_SIX, moe4.workspace(moe4.moe4_workspace_size(moe4.OP_HADAMARD_QUANT)))
    row_d, w_d = to_dev(row_of), to_dev(w)
    y = torch.empty((T, d), dtype=torch.int16, device=DEV)
    moe4.moe4_combine_hadamard(c, s, g, row_d, w_d, T, k, d, y)
    yhat = torch.empty((R, d), dtype=torch.int16, device=DEV)
    moe4.hadamard_dequant(c, s, g, R, d, yhat)
    y2 = torch.empty((T, d), dtype=torch.int16, device=DEV)
    moe4.moe4_combine(yhat, row_d, w_d, T, k, d, y2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    if T <= 1024:
        rh = oracle.hadamard_dequant(to_np(c), to_np(s), to_np(g)[0])
        assert np.array_equal(to_np(y, np.uint16), oracle.combine(rh, row_of, w))
