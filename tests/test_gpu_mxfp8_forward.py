"""GPU parity of the MXFP8 forward pass kept for the final layers ("Inkling 2 Small's Native 4-Bit
Training: Debut and Doubts", "Confirmed" list; "Thinking Machines: Nvidia FP4 Up to 6x Faster,
Runs Gain 8%"): bf16 activations and weights quantised to MXFP8 with nearest-even (E4M3, E8M0
per 32 by the ceiling rule), the activation rows gathered into expert order, and the rows-grouped
MXFP8 GEMM for gate/up (binary32 out) and down (bf16 out).

Quantised operands and the gather are compared bit for bit; the GEMMs use the tolerance of the
other grouped-GEMM tests (relative Frobenius <= 1e-5 and |D - D_ref| <= 2^-16 * sum |a*b| per
element; bf16 output adds one bf16 rounding).  Inputs: the small grouped MoE (T = 4096, d = 2048,
f = 1024, 8 experts, top-2) in full, and the Inkling-shaped layer (T = 16384, d = 4096, f = 2048,
384 experts, top-8) on sampled rows of three experts.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import inputs, moe4
from gpu_helpers import DEV, empty_u8, first_mismatch, to_dev, to_np
from test_gpu_gemm import check_bf16, check_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    moe4.load()


def _mx_rows(x_dev, rows, cols):
    q = empty_u8(rows, cols)
    e8 = empty_u8(rows, cols // 32)
    moe4.mxfp8_quantize(x_dev, rows, cols, q, e8, 0, 0, moe4.ROWWISE)
    return q, e8


def _plan(idx_np, T, k, E):
    rows_cap = T * k + 127 * E
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_of = torch.empty((T, k), dtype=torch.int32, device=DEV)
    src_of = torch.empty(rows_cap, dtype=torch.int32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_PERMUTE_PLAN, T, k, E))
    moe4.moe4_permute_plan(to_dev(idx_np), T, k, E, offs, row_of, src_of, rows_cap, ws)
    return offs, src_of


def _gather_mx(q, e8, T, cols, src_of, Rp):
    oq, oe = empty_u8(Rp, cols), empty_u8(Rp, cols // 32)
    moe4.moe4_permute_nvfp4(q, e8, T, cols, src_of, Rp, oq, oe, moe4.MXFP8)
    return oq, oe


def _gemm(aq, ae, bq, be, offs, E, M, N, K, out_bf16=False):
    D = torch.empty((M, N), dtype=torch.int16 if out_bf16 else torch.float32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, E, N, K))
    flags = (moe4.OUT_BF16 if out_bf16 else moe4.OUT_F32) | moe4.GROUP_M
    moe4.grouped_gemm_mxfp8(aq, ae, bq, be, offs, E, M, N, K, D, flags, ws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    return D


def test_mxfp8_gather_with_padding():
    T, E, k, cols = 37, 5, 2, 96
    rng = np.random.default_rng(3)
    idx, _ = oracle.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
    x = inputs.to_bf16_bits(rng.standard_normal((T, cols)).astype(np.float32))
    q, e8 = _mx_rows(to_dev(x), T, cols)
    offs, src_of = _plan(idx, T, k, E)
    roffs, rrow = oracle.permute_plan(idx, E)
    Rp = int(roffs[-1])
    oq, oe = _gather_mx(q, e8, T, cols, src_of, Rp)
    torch.cuda.synchronize()
    rq, re = oracle.mxfp8_quantize(oracle.bf16_to_f32(x), colwise=False)
    assert first_mismatch(to_np(oq), oracle.permute_rows(rq, rrow, Rp)) is None
    assert first_mismatch(to_np(oe), oracle.permute_rows(re, rrow, Rp)) is None


def test_mxfp8_forward_small_moe():
    T, d, f, E, k = 4096, 2048, 1024, 8, 2
    rng = np.random.default_rng(31)
    idx, _ = oracle.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
    x = inputs.to_bf16_bits((rng.standard_t(3, (T, d)) / np.sqrt(3)).astype(np.float32))
    w_gu = inputs.to_bf16_bits((rng.standard_normal((E * 2 * f, d)) * 0.02).astype(np.float32))
    w_d = inputs.to_bf16_bits((rng.standard_normal((E * d, f)) * 0.02).astype(np.float32))
    roffs, rrow = oracle.permute_plan(idx, E)
    Rp = int(roffs[-1])
    h = inputs.to_bf16_bits(rng.standard_normal((Rp, f)).astype(np.float32))

    offs, src_of = _plan(idx, T, k, E)
    xq, xe = _mx_rows(to_dev(x), T, d)
    xpq, xpe = _gather_mx(xq, xe, T, d, src_of, Rp)
    gq, ge = _mx_rows(to_dev(w_gu), E * 2 * f, d)
    GU = _gemm(xpq, xpe, gq, ge, offs, E, Rp, 2 * f, d)
    hq, he = _mx_rows(to_dev(h), Rp, f)
    dq, de = _mx_rows(to_dev(w_d), E * d, f)
    Y = _gemm(hq, he, dq, de, offs, E, Rp, d, f, out_bf16=True)

    rxq, rxe = oracle.mxfp8_quantize(oracle.bf16_to_f32(x), colwise=False)
    rpq, rpe = oracle.permute_rows(rxq, rrow, Rp), oracle.permute_rows(rxe, rrow, Rp)
    assert first_mismatch(to_np(xpq), rpq) is None and first_mismatch(to_np(xpe), rpe) is None
    rgq, rge = oracle.mxfp8_quantize(oracle.bf16_to_f32(w_gu), colwise=False)
    assert first_mismatch(to_np(gq), rgq) is None and first_mismatch(to_np(ge), rge) is None
    Dref, S = oracle.grouped_gemm_m(oracle.mxfp8_dequantize(rpq, rpe),
                                    oracle.mxfp8_dequantize(rgq, rge).reshape(E, 2 * f, d), roffs)
    check_f32(to_np(GU), Dref, S, "mxfp8 forward gate/up")
    rhq, rhe = oracle.mxfp8_quantize(oracle.bf16_to_f32(h), colwise=False)
    rdq, rde = oracle.mxfp8_quantize(oracle.bf16_to_f32(w_d), colwise=False)
    Yref, SY = oracle.grouped_gemm_m(oracle.mxfp8_dequantize(rhq, rhe),
                                     oracle.mxfp8_dequantize(rdq, rde).reshape(E, d, f), roffs)
    check_bf16(to_np(Y, np.uint16), Yref, SY)


def test_mxfp8_forward_gate_up_full_size_sampled_rows():
    T, d, f, E, k = 16384, 4096, 2048, 384, 8
    rng = np.random.default_rng(0)
    lg = (rng.standard_normal((T, E)) + rng.standard_normal(E)).astype(np.float32)
    idx, _ = oracle.route_topk(lg, k)
    roffs, rrow = oracle.permute_plan(idx, E)
    Rp = int(roffs[-1])
    x = inputs.device_student_t((T, d), inputs.device_generator(6, 0, DEV), DEV).view(torch.int16)
    w = inputs.device_normal((E * 2 * f, d), 0.02, inputs.device_generator(6, 1, DEV), DEV).view(torch.int16)

    offs, src_of = _plan(idx, T, k, E)
    xq, xe = _mx_rows(x, T, d)
    xpq, xpe = _gather_mx(xq, xe, T, d, src_of, Rp)
    del xq, xe
    gq, ge = _mx_rows(w, E * 2 * f, d)
    GU = _gemm(xpq, xpe, gq, ge, offs, E, Rp, 2 * f, d)
    del gq, ge

    src = np.full(Rp, -1, np.int64)
    src[rrow.reshape(-1)] = np.repeat(np.arange(T), k)
    sizes = np.diff(roffs)
    for e in [int(np.argmax(sizes)), int(np.nonzero(sizes)[0][0]), int(np.nonzero(sizes)[0][-1])]:
        lo, hi = int(roffs[e]), int(roffs[e + 1])
        rows = np.unique(np.concatenate([np.random.default_rng(e).choice(np.arange(lo, hi), 12), [lo, hi - 1]]))
        real = src[rows] >= 0
        xs = np.zeros((len(rows), d), np.uint16)
        xs[real] = to_np(x[torch.as_tensor(src[rows][real], device=DEV)], np.uint16)
        rxq, rxe = oracle.mxfp8_quantize(oracle.bf16_to_f32(xs), colwise=False)
        we = oracle.bf16_to_f32(to_np(w[e * 2 * f:(e + 1) * 2 * f], np.uint16))
        rwq, rwe = oracle.mxfp8_quantize(we, colwise=False)
        Dref, S = oracle.grouped_gemm_m(oracle.mxfp8_dequantize(rxq, rxe),
                                        oracle.mxfp8_dequantize(rwq, rwe)[None], np.array([0, len(rows)]))
        check_f32(to_np(GU[torch.as_tensor(rows, device=DEV)]), Dref, S, "expert %d" % e)
