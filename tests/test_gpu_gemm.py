"""GPU parity of the block-scaled grouped GEMMs against the oracle's float64 GEMM of the operands
the oracle quantised itself.

Tolerance (binary32 output): relative Frobenius error <= 1e-5 and, element by element,
|D - D_ref| <= 2^-16 * sum_k |a_k * b_k|.  bf16 output: within one bf16 ulp of RN_bf16(D_ref).
The NVFP4 GEMM is the expert forward ("Inkling 2 Small's Native 4-Bit Training: Debut and Doubts",
"Confirmed": NVFP4 forward of the expert layers with dedicated kernels); the MXFP8 GEMMs are the
backward dgrad (rows grouped by expert) and wgrad (contraction grouped by expert).
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import inputs, moe4
from gpu_helpers import DEV, empty_u8, mma_layout, nvfp4_quantize, to_dev, to_np

pytestmark = pytest.mark.gpu

REL_FRO = 1e-5
ELEM = 2.0 ** -16


def check_f32(D, Dref, S, what=""):
    D = D.astype(np.float64)
    err = np.abs(D - Dref)
    nref = np.linalg.norm(Dref)
    rel = np.linalg.norm(D - Dref) / (nref if nref > 0 else 1.0)
    bad = err > ELEM * S
    assert rel <= REL_FRO and not bad.any(), (
        "%s rel_fro=%.3e, %d of %d elements over 2^-16*S, worst err/S=%.3e, D[0,:4]=%s ref=%s" %
        (what, rel, int(bad.sum()), bad.size, float(np.max(err / np.maximum(S, 1e-300))),
         D.reshape(-1)[:4], Dref.reshape(-1)[:4]))


def check_bf16(Dbits, Dref, S):
    """bf16 output: one bf16 rounding (at most one ulp, 2^-8 relative) on top of the binary32
    accumulation bound; near cancellation the accumulation term dominates."""
    got = oracle.bf16_to_f32(Dbits).astype(np.float64)
    bad = np.abs(got - Dref) > 2.0 ** -8 * np.abs(Dref) + ELEM * S
    assert not bad.any(), "%d of %d bf16 outputs outside one ulp + 2^-16*S" % (int(bad.sum()), bad.size)


def _bf16(rng, shape, std=1.0, t=False):
    x = rng.standard_t(3, shape) / np.sqrt(3) if t else rng.standard_normal(shape)
    return inputs.to_bf16_bits((x * std).astype(np.float32))


def _offs(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _nvfp4_case(rows_sizes, N, K, seed, out_bf16=False, sf_mma=False):
    rng = np.random.default_rng(seed)
    E = len(rows_sizes)
    offs = _offs(rows_sizes)
    R = int(offs[-1])
    a_bits = _bf16(rng, (R, K), t=True)
    b_bits = _bf16(rng, (E * N, K), 0.02)
    # device path
    ac, asf, ag = nvfp4_quantize(to_dev(a_bits), 1, R, K)
    bc, bsf, bg = nvfp4_quantize(to_dev(b_bits), E, N, K)
    flags = moe4.OUT_BF16 if out_bf16 else moe4.OUT_F32
    if sf_mma:
        asf2, bsf2 = torch.empty_like(asf), torch.empty_like(bsf)
        moe4.moe4_sf_to_mma_layout(asf, 1, R, K // 16, asf2)
        moe4.moe4_sf_to_mma_layout(bsf, E, N, K // 16, bsf2)
        asf, bsf = asf2, bsf2
        flags |= moe4.SF_MMA_LAYOUT
    D = torch.empty((R, N), dtype=torch.int16 if out_bf16 else torch.float32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(0, R, E, N, K))
    moe4.grouped_expert_gemm_nvfp4(ac, asf, ag, bc, bsf, bg, to_dev(offs), E, R, N, K, D, flags, ws)
    assert moe4.moe4_get_status() == moe4.OK
    # oracle path
    rac, ras, rag = oracle.nvfp4_quantize(oracle.bf16_to_f32(a_bits))
    rbc, rbs, rbg = oracle.nvfp4_quantize(oracle.bf16_to_f32(b_bits).reshape(E, N, K))
    if not sf_mma:  # the operands themselves must already agree bit for bit
        for got, want, name in ((ac, rac, "A codes"), (asf, ras, "A scales"), (ag, rag, "A g_dec"),
                                (bc, rbc, "B codes"), (bsf, rbs, "B scales"), (bg, rbg, "B g_dec")):
            g_np = to_np(got).reshape(np.shape(want))
            assert np.array_equal(g_np, want), "%s differ in %d places" % (name, int(np.sum(g_np != want)))
    Dref, S = oracle.grouped_gemm_m(oracle.nvfp4_dequantize(rac, ras, rag),
                                    oracle.nvfp4_dequantize(rbc, rbs, rbg), offs)
    return D, Dref, S


def test_nvfp4_single_expert_workload():
    # X 256x512 (N(0,1) with 1% outliers x20) times W (512x256 stored K-major as 256x512)
    rng = inputs.host_rng(1, 0)
    x = inputs.to_bf16_bits(inputs.host_outliers(rng, inputs.host_normal(rng, (256, 512))))
    w = inputs.to_bf16_bits(inputs.host_normal(inputs.host_rng(1, 1), (256, 512), 0.02))
    ac, asf, ag = nvfp4_quantize(to_dev(x), 1, 256, 512)
    bc, bsf, bg = nvfp4_quantize(to_dev(w), 1, 256, 512)
    offs = to_dev(np.array([0, 256], np.int32))
    D = torch.empty((256, 256), dtype=torch.float32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(0, 256, 1, 256, 512))
    moe4.grouped_expert_gemm_nvfp4(ac, asf, ag, bc, bsf, bg, offs, 1, 256, 256, 512, D, moe4.OUT_F32, ws)
    assert moe4.moe4_get_status() == moe4.OK
    rac, ras, rag = oracle.nvfp4_quantize(oracle.bf16_to_f32(x))
    rbc, rbs, rbg = oracle.nvfp4_quantize(oracle.bf16_to_f32(w))
    Dref, S = oracle.grouped_gemm_m(oracle.nvfp4_dequantize(rac, ras, rag),
                                    oracle.nvfp4_dequantize(rbc, rbs, rbg)[None], np.array([0, 256]))
    check_f32(to_np(D), Dref, S, "single expert")


@pytest.mark.parametrize("sf_mma", [False, True])
def test_nvfp4_grouped_with_empty_groups(sf_mma):
    D, Dref, S = _nvfp4_case([128, 0, 256, 384, 128, 0], N=512, K=768, seed=5, sf_mma=sf_mma)
    check_f32(to_np(D), Dref, S, "grouped")


def test_nvfp4_bf16_output():
    D, Dref, S = _nvfp4_case([256, 128], N=256, K=512, seed=6, out_bf16=True)
    check_bf16(to_np(D, np.uint16), Dref, S)


def test_nvfp4_small_moe_shapes():
    # 8 experts, d_model 2048, gate/up width 2048 (2 x 1024): groups of a top-2 routing, padded
    rng = np.random.default_rng(12)
    counts = rng.multinomial(8192, np.ones(8) / 8)
    sizes = (counts + 127) // 128 * 128
    D, Dref, S = _nvfp4_case(list(sizes), N=2048, K=2048, seed=13)
    check_f32(to_np(D), Dref, S, "small moe")


def _mxfp8_rowwise(x_bits, rows, cols):
    q = empty_u8(rows, cols)
    e8 = empty_u8(rows, cols // 32)
    moe4.mxfp8_quantize(to_dev(x_bits), rows, cols, q, e8, 0, 0, moe4.ROWWISE)
    return q, e8


def test_mxfp8_dgrad_group_m():
    rng = np.random.default_rng(21)
    sizes = [256, 0, 128, 384]
    E, N, K = len(sizes), 512, 640
    offs = _offs(sizes)
    M = int(offs[-1])
    a_bits = _bf16(rng, (M, K))
    b_bits = _bf16(rng, (E * N, K), 0.02)
    aq, ae = _mxfp8_rowwise(a_bits, M, K)
    bq, be = _mxfp8_rowwise(b_bits, E * N, K)
    D = torch.empty((M, N), dtype=torch.float32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, E, N, K))
    moe4.grouped_gemm_mxfp8(aq, ae, bq, be, to_dev(offs), E, M, N, K, D, moe4.OUT_F32 | moe4.GROUP_M, ws)
    assert moe4.moe4_get_status() == moe4.OK
    ra = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(oracle.bf16_to_f32(a_bits), colwise=False))
    rb = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(oracle.bf16_to_f32(b_bits), colwise=False))
    Dref, S = oracle.grouped_gemm_m(ra, rb.reshape(E, N, K), offs)
    check_f32(to_np(D), Dref, S, "mxfp8 dgrad")


@pytest.mark.parametrize("accumulate", [False, True])
def test_mxfp8_wgrad_group_k(accumulate):
    rng = np.random.default_rng(22)
    sizes = [128, 256, 0, 384]
    E, M, N = len(sizes), 256, 512
    offs = _offs(sizes)
    Kt = int(offs[-1])
    a_bits = _bf16(rng, (M, Kt))
    b_bits = _bf16(rng, (N, Kt))
    aq, ae = _mxfp8_rowwise(a_bits, M, Kt)
    bq, be = _mxfp8_rowwise(b_bits, N, Kt)
    init = rng.standard_normal((E, M, N)).astype(np.float32)
    D = to_dev(init) if accumulate else torch.full((E, M, N), np.nan, dtype=torch.float32, device=DEV)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, 1, N, Kt))
    flags = moe4.OUT_F32 | moe4.GROUP_K | (moe4.ACCUMULATE if accumulate else 0)
    moe4.grouped_gemm_mxfp8(aq, ae, bq, be, to_dev(offs), E, M, N, Kt, D, flags, ws)
    assert moe4.moe4_get_status() == moe4.OK
    ra = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(oracle.bf16_to_f32(a_bits), colwise=False))
    rb = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(oracle.bf16_to_f32(b_bits), colwise=False))
    Dref, S = oracle.grouped_gemm_k(ra, rb, offs)
    got = to_np(D)
    if accumulate:
        # D = RN(init + product): widen the bound by the rounding of that one addition
        Dref = Dref + init
        S = S + np.abs(init) * 2.0 ** -7
    check_f32(got, Dref, S, "mxfp8 wgrad")
    if not accumulate:
        assert np.all(got[2] == 0)


@pytest.mark.parametrize("sizes,M,N", [([128, 256, 0, 384], 256, 512),
                                         ([128, 128, 0, 512, 256, 128, 384, 128], 1024, 2048),
                                         ([128, 0, 256], 256, 512),
                                         ([256, 128, 0], 128, 512)])
def test_mxfp8_wgrad_fused_sgd_equals_gemm_then_sgd(sizes, M, N):
    """The fused weight-gradient + SGD epilogue is bit-identical to the unfused pair, and its
    per-expert amax equals max |bf16 copy|.  The second case has 1024 output tiles, several per
    CTA, so each CTA's epilogue also prefetches the master weights of its next tile.  The grid is
    one CTA per tile up to one per SM, so the tile schedule takes both forms an even grid can
    take: every third slot on the front of the size-sorted list (grids of 32 and 148 CTAs) and
    alternating (24 and 12 CTAs, multiples of 3).  Tile counts are even (N is a multiple of 256),
    so the list-in-order form, for odd multiples of 3, needs an odd SM count."""
    rng = np.random.default_rng(23)
    E = len(sizes)
    offs = _offs(sizes)
    Kt = int(offs[-1])
    aq, ae = _mxfp8_rowwise(_bf16(rng, (M, Kt)), M, Kt)
    bq, be = _mxfp8_rowwise(_bf16(rng, (N, Kt)), N, Kt)
    w0 = (rng.standard_normal((E, M, N)) * 0.02).astype(np.float32)
    lr = 1e-2
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, 1, N, Kt))
    # unfused: dW to memory, then SGD
    dW = torch.empty((E, M, N), dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8(aq, ae, bq, be, to_dev(offs), E, M, N, Kt, dW, moe4.OUT_F32 | moe4.GROUP_K, ws)
    w_ref = to_dev(w0)
    wb_ref = torch.empty((E, M, N), dtype=torch.int16, device=DEV)
    moe4.moe4_sgd_update(w_ref, dW, w_ref.numel(), lr, wb_ref)
    # fused
    w_f = to_dev(w0)
    wb_f = to_dev(oracle.f32_to_bf16(w0))          # the bf16 copy that goes with w0
    amax = torch.full((E,), -1.0, dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8_wgrad_sgd(aq, ae, bq, be, to_dev(offs), E, M, N, Kt, w_f, wb_f, lr, amax, 0, ws)
    assert moe4.moe4_get_status() == moe4.OK
    torch.cuda.synchronize()
    assert torch.equal(w_f, w_ref)
    assert torch.equal(wb_f, wb_ref)
    want = np.abs(oracle.bf16_to_f32(to_np(wb_ref, np.uint16))).reshape(E, -1).max(axis=1)
    want[np.asarray(sizes) == 0] = -1.0  # experts without rows are skipped: amax left as it was
    assert np.array_equal(to_np(amax), want.astype(np.float32))
    # without a bf16 copy: the same master weights and amax
    w_n = to_dev(w0)
    amax_n = torch.full((E,), -1.0, dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8_wgrad_sgd(aq, ae, bq, be, to_dev(offs), E, M, N, Kt, w_n, None, lr, amax_n, 0, ws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    assert torch.equal(w_n, w_ref) and torch.equal(amax_n, amax)


def test_mxfp8_gemms_read_tile_layout_scales():
    """MOE4_SF_MMA_LAYOUT on the MXFP8 GEMMs (operand scales already in the tensor-core tile
    layout, as the producers write them with MOE4_SF_OUT_MMA): the same bits as from canonical
    scales, for the rows-grouped dgrad and the contraction-grouped fused SGD."""
    rng = np.random.default_rng(24)
    sizes = [256, 0, 128, 384]
    E, N, K = len(sizes), 512, 640
    offs = to_dev(_offs(sizes))
    M = int(sum(sizes))
    aq, ae = _mxfp8_rowwise(_bf16(rng, (M, K)), M, K)
    bq, be = _mxfp8_rowwise(_bf16(rng, (E * N, K), 0.02), E * N, K)
    ae_t, be_t = mma_layout(ae, M, K // 32), mma_layout(be, E * N, K // 32)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, E, N, K))
    D0 = torch.empty((M, N), dtype=torch.float32, device=DEV)
    D1 = torch.empty((M, N), dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8(aq, ae, bq, be, offs, E, M, N, K, D0, moe4.OUT_F32 | moe4.GROUP_M, ws)
    moe4.grouped_gemm_mxfp8(aq, ae_t, bq, be_t, offs, E, M, N, K, D1, moe4.OUT_F32 | moe4.GROUP_M | moe4.SF_MMA_LAYOUT,
                            None)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    assert torch.equal(D0, D1)
    # contraction-grouped with the fused update: A [Mw, Kt], B [Nw, Kt]
    Mw, Nw, Kt = 256, 512, M
    xq, xe = _mxfp8_rowwise(_bf16(rng, (Mw, Kt)), Mw, Kt)
    yq, ye = _mxfp8_rowwise(_bf16(rng, (Nw, Kt)), Nw, Kt)
    w0 = to_dev((rng.standard_normal((E, Mw, Nw)) * 0.02).astype(np.float32))
    outs = []
    for tile in (False, True):
        w, wb = w0.clone(), torch.zeros((E, Mw, Nw), dtype=torch.int16, device=DEV)
        amax = torch.full((E,), -1.0, dtype=torch.float32, device=DEV)
        a_e = mma_layout(xe, Mw, Kt // 32) if tile else xe
        b_e = mma_layout(ye, Nw, Kt // 32) if tile else ye
        gws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, Mw, 1, Nw, Kt))
        moe4.grouped_gemm_mxfp8_wgrad_sgd(xq, a_e, yq, b_e, offs, E, Mw, Nw, Kt, w, wb, 1e-2, amax,
                                          moe4.SF_MMA_LAYOUT if tile else 0, gws)
        torch.cuda.synchronize()
        assert moe4.moe4_get_status() == moe4.OK
        outs.append((w, wb, amax))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_nvfp4_forward_gate_up_full_size_sampled_rows():
    """The layer step's gate/up GEMM as it runs there: 16384 tokens x d_model 4096 (Student-t(3))
    quantised to NVFP4 with one per-tensor scale, gathered into expert order by a top-8 plan over
    384 experts (N(0,1) logits + per-expert bias), tile-layout scales, against 384 experts'
    gate/up weights [4096, 4096] N(0, 0.02) with per-expert scales; binary32 output.  Checked on
    sampled rows of three experts (the largest group, the first and the last non-empty one): the
    oracle quantises those token rows with the tensor's amax and the expert's weights with the
    expert's amax, and multiplies in float64."""
    T, d, f, E, k = 16384, 4096, 2048, 384, 8
    rng = np.random.default_rng(0)
    lg = (rng.standard_normal((T, E)) + rng.standard_normal(E)).astype(np.float32)
    idx, _ = oracle.route_topk(lg, k)
    roffs, rrow = oracle.permute_plan(idx, E)
    Rp = int(roffs[-1])
    rows_cap = T * k + 127 * E
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_of = torch.empty((T, k), dtype=torch.int32, device=DEV)
    src_of = torch.empty(rows_cap, dtype=torch.int32, device=DEV)
    moe4.moe4_permute_plan(to_dev(idx), T, k, E, offs, row_of, src_of, rows_cap,
                           moe4.workspace(moe4.moe4_workspace_size(moe4.OP_PERMUTE_PLAN, T, k, E)))
    x = inputs.device_student_t((T, d), inputs.device_generator(21, 0, DEV), DEV).view(torch.int16)
    w = inputs.device_normal((E * 2 * f, d), 0.02, inputs.device_generator(21, 1, DEV), DEV).view(torch.int16)
    xc, xs, xg = nvfp4_quantize(x, 1, T, d)
    xpc, xps = empty_u8(Rp, d // 2), empty_u8(Rp, d // 16)
    moe4.moe4_permute_nvfp4(xc, xs, T, d, src_of, Rp, xpc, xps, moe4.SF_MMA_LAYOUT)
    del xc, xs
    wc, ws_, wg = nvfp4_quantize(w, E, 2 * f, d, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT)
    GU = torch.empty((Rp, 2 * f), dtype=torch.float32, device=DEV)
    gws = moe4.workspace(moe4.moe4_workspace_size_gemm(0, Rp, E, 2 * f, d))
    moe4.grouped_expert_gemm_nvfp4(xpc, xps, xg, wc, ws_, wg, offs, E, Rp, 2 * f, d, GU,
                                   moe4.OUT_F32 | moe4.SF_MMA_LAYOUT, gws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    assert np.array_equal(to_np(offs), roffs)
    del wc, ws_

    x32 = oracle.bf16_to_f32(to_np(x, np.uint16))
    x_amax = np.abs(x32).max()
    src = np.full(Rp, -1, np.int64)
    src[rrow.reshape(-1)] = np.repeat(np.arange(T), k)
    sizes = np.diff(roffs)
    live = np.nonzero(sizes)[0]
    for e in [int(np.argmax(sizes)), int(live[0]), int(live[-1])]:
        lo, hi = int(roffs[e]), int(roffs[e + 1])
        rows = np.unique(np.concatenate([np.random.default_rng(e).choice(np.arange(lo, hi), 12), [lo, hi - 1]]))
        real = src[rows] >= 0
        xs_ = np.zeros((len(rows), d), np.float32)
        xs_[real] = x32[src[rows][real]]
        rxc, rxs, rxg = oracle.nvfp4_quantize(xs_, amax=x_amax)
        we = oracle.bf16_to_f32(to_np(w[e * 2 * f:(e + 1) * 2 * f], np.uint16))
        rwc, rws, rwg = oracle.nvfp4_quantize(we)
        Dref, S = oracle.grouped_gemm_m(oracle.nvfp4_dequantize(rxc, rxs, rxg),
                                        oracle.nvfp4_dequantize(rwc, rws, rwg)[None], np.array([0, len(rows)]))
        check_f32(to_np(GU[torch.as_tensor(rows, device=DEV)]), Dref, S, "expert %d" % e)


def test_mxfp8_wgrad_fused_sgd_full_size_equals_unfused():
    """The layer step's down-projection weight update at full size: 384 experts, W32 [384, 4096,
    2048], the contraction over each expert's rows of a skewed top-8 routing (largest group
    thousands of rows, many tiny, some empty), MXFP8 operands with tile-layout scales.  The fused
    kernel without a bf16 copy (size-interleaved tile schedule, five-buffer ring) gives the same
    FP32 masters as the contraction-grouped GEMM to memory followed by moe4_sgd_update, bit for
    bit, and the amax of their bf16 rounding."""
    E, M, N = 384, 4096, 2048
    rng = np.random.default_rng(1)
    counts = rng.multinomial(16384 * 8, rng.dirichlet(np.ones(E) * 0.5))
    offs_np = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    Kt = int(offs_np[-1])
    offs = to_dev(offs_np)
    gen = inputs.device_generator(23, 0, DEV)

    def codes(n):  # E4M3 codes without the NaN patterns
        c = torch.randint(0, 0x7F, (n,), generator=gen, device=DEV, dtype=torch.int32)
        s = torch.randint(0, 2, (n,), generator=gen, device=DEV, dtype=torch.int32) * 0x80
        return (c | s).to(torch.uint8)

    a, b = codes(M * Kt), codes(N * Kt)
    ae = torch.randint(118, 124, (M * Kt // 32,), generator=gen, device=DEV, dtype=torch.int32).to(torch.uint8)
    be = torch.randint(118, 124, (N * Kt // 32,), generator=gen, device=DEV, dtype=torch.int32).to(torch.uint8)
    ae_t, be_t = mma_layout(ae, M, Kt // 32), mma_layout(be, N, Kt // 32)
    w0 = inputs.device_normal((E, M, N), 0.02, inputs.device_generator(23, 1, DEV), DEV, dtype=torch.float32)
    lr = 1e-3
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, 1, N, Kt))
    dW = torch.empty((E, M, N), dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8(a, ae, b, be, offs, E, M, N, Kt, dW, moe4.OUT_F32 | moe4.GROUP_K, ws)
    w_ref = w0.clone()
    wb_ref = torch.empty((E, M, N), dtype=torch.int16, device=DEV)
    moe4.moe4_sgd_update(w_ref, dW, w_ref.numel(), lr, wb_ref)
    del dW
    w_f = w0.clone()
    amax = torch.full((E,), -1.0, dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8_wgrad_sgd(a, ae_t, b, be_t, offs, E, M, N, Kt, w_f, None, lr, amax, moe4.SF_MMA_LAYOUT,
                                      ws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    assert torch.equal(w_f, w_ref)
    want = wb_ref.view(torch.bfloat16).abs().reshape(E, -1).amax(dim=1).float()
    want[torch.as_tensor(counts == 0, device=DEV)] = -1.0  # experts without rows are skipped
    assert torch.equal(amax, want)


@pytest.mark.parametrize("M,N", [(4096, 2048), (4096, 4096)])
def test_mxfp8_wgrad_full_contraction_against_oracle(M, N):
    """The contraction-grouped weight gradient at the layer's contraction lengths, against the
    oracle: groups of 9728 rows (the size of the largest expert group of the layer step's skewed
    routing), 1152 rows, one 128-row tile, an empty group and 256 rows, each ending in zero padding
    rows.  A = the column-wise MXFP8 (nearest-even) of a bf16 gradient [Kt, M] (dY for the down
    projection, dGU for gate/up); B = the dequantise -> transpose -> MXFP8 stochastic-rounding
    requantisation of an NVFP4 forward operand [Kt, N] (H, or the gathered X).  Both operands are
    first checked bit for bit against the oracle's own quantisation, then the binary32 dW is
    compared element by element on 40 sampled rows of M (every column, the full contraction of
    each group) with the oracle's float64 product, and the fused SGD update on the same operands
    against the oracle's sgd_update of that product ("4-bit computation from the start of Inkling 2
    Small's pretraining", backward-pass paragraphs; precisions paragraph: FP32 master weights)."""
    sizes = [9728, 1152, 128, 0, 256]
    pads = [37, 100, 5, 0, 128 - 77]
    E = len(sizes)
    offs_np = _offs(sizes)
    Kt = int(offs_np[-1])
    rng = np.random.default_rng(40 + N // 1024)
    live = np.ones(Kt, bool)
    for lo, sz, pd in zip(offs_np[:-1], sizes, pads):
        live[lo + sz - pd:lo + sz] = False
    g_bits = _bf16(rng, (Kt, M))
    x_bits = _bf16(rng, (Kt, N), t=True)
    g_bits[~live] = 0
    x_bits[~live] = 0
    # device operands
    aq, ae = empty_u8(M, Kt), empty_u8(M, Kt // 32)
    moe4.mxfp8_quantize(to_dev(g_bits), Kt, M, aq, ae, 0, 0, moe4.COLWISE)
    xc, xs, xg = nvfp4_quantize(to_dev(x_bits), 1, Kt, N)
    bq, be = empty_u8(N, Kt), empty_u8(N, Kt // 32)
    moe4.mxfp8_requant_transpose_sr(xc, xs, xg, 1, Kt, N, bq, be, 9, 2, moe4.SR)
    # oracle operands, and the device's equal to them bit for bit
    raq, rae = oracle.mxfp8_quantize(oracle.bf16_to_f32(g_bits), colwise=True)
    rxc, rxs, rxg = oracle.nvfp4_quantize(oracle.bf16_to_f32(x_bits))
    rbq, rbe = oracle.mxfp8_requant_transpose(rxc, rxs, rxg, sr=True, seed=9, stream_id=2)
    for got, want, name in ((aq, raq, "A codes"), (ae, rae, "A scales"), (bq, rbq, "B codes"), (be, rbe, "B scales")):
        g_np = to_np(got).reshape(want.shape)
        assert np.array_equal(g_np, want), "%s differ in %d places" % (name, int(np.sum(g_np != want)))
    offs = to_dev(offs_np)
    ae_t, be_t = mma_layout(ae, M, Kt // 32), mma_layout(be, N, Kt // 32)
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, 1, N, Kt))
    D = torch.full((E, M, N), np.nan, dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8(aq, ae_t, bq, be_t, offs, E, M, N, Kt, D, moe4.OUT_F32 | moe4.GROUP_K | moe4.SF_MMA_LAYOUT,
                            None)
    w0 = inputs.device_normal((E, M, N), 0.02, inputs.device_generator(40, N, DEV), DEV, dtype=torch.float32)
    lr = 1e-3
    w = w0.clone()
    amax = torch.full((E,), -1.0, dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8_wgrad_sgd(aq, ae_t, bq, be_t, offs, E, M, N, Kt, w, None, lr, amax, moe4.SF_MMA_LAYOUT,
                                      ws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    rows = np.unique(np.concatenate([np.random.default_rng(N).choice(M, 38, replace=False), [0, M - 1]]))
    rows_d = torch.as_tensor(rows, device=DEV)
    ra = oracle.mxfp8_dequantize(raq, rae)[rows]
    rb = oracle.mxfp8_dequantize(rbq, rbe)
    Dref, S = oracle.grouped_gemm_k(ra, rb, offs_np)
    Dg = to_np(D[:, rows_d])
    for e in range(E):
        check_f32(Dg[e], Dref[e], S[e], "wgrad expert %d (%d rows)" % (e, sizes[e]))
    assert np.all(Dg[3] == 0)
    # the fused update against the oracle's SGD of the oracle's product: the product's error
    # (2^-16 * S, times lr) plus one rounding of the step and one of the difference
    w0_np = to_np(w0[:, rows_d])
    w_ref, _ = oracle.sgd_update(w0_np, Dref.astype(np.float32), lr)
    got = to_np(w[:, rows_d]).astype(np.float64)
    tol = lr * ELEM * S + 2.0 ** -23 * (lr * np.abs(Dref) + np.abs(w_ref.astype(np.float64)))
    bad = np.abs(got - w_ref) > tol
    assert not bad.any(), "%d of %d updated weights outside the bound" % (int(bad.sum()), bad.size)
    assert torch.equal(w[3], w0[3])  # the empty group keeps its weights
    want_amax = torch.stack([w[e].to(torch.bfloat16).abs().max().float() for e in range(E)])
    want_amax[3] = -1.0  # and its amax entry is not written
    assert torch.equal(amax, want_amax)


def test_nvfp4_down_bf16_full_size_sampled_rows():
    """The layer step's down-projection GEMM as it runs there: H [padded rows, 2048] (Student-t(3),
    zero on the padding rows of a top-8 plan over 384 experts) quantised to NVFP4 with one
    per-tensor scale, times 384 experts' down weights [4096, 2048] N(0, 0.02) with per-expert
    scales, tile-layout scales, bf16 output.  Checked on sampled rows of three experts (the largest
    group, the first and the last non-empty one) against the oracle's float64 product of its own
    quantisation (H rows with the whole tensor's amax, each expert's weights with its own)."""
    T, d, f, E, k = 16384, 4096, 2048, 384, 8
    rng = np.random.default_rng(0)
    lg = (rng.standard_normal((T, E)) + rng.standard_normal(E)).astype(np.float32)
    idx, _ = oracle.route_topk(lg, k)
    roffs, rrow = oracle.permute_plan(idx, E)
    Rp = int(roffs[-1])
    real = np.zeros(Rp, bool)
    real[rrow.reshape(-1)] = True
    h = inputs.device_student_t((Rp, f), inputs.device_generator(22, 0, DEV), DEV).view(torch.int16)
    h[torch.as_tensor(~real, device=DEV)] = 0
    w = inputs.device_normal((E * d, f), 0.02, inputs.device_generator(22, 1, DEV), DEV).view(torch.int16)
    hc, hs, hg = nvfp4_quantize(h, 1, Rp, f, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT)
    wc, wsf, wg = nvfp4_quantize(w, E, d, f, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT)
    Y = torch.empty((Rp, d), dtype=torch.int16, device=DEV)
    gws = moe4.workspace(moe4.moe4_workspace_size_gemm(0, Rp, E, d, f))
    moe4.grouped_expert_gemm_nvfp4(hc, hs, hg, wc, wsf, wg, to_dev(roffs), E, Rp, d, f, Y,
                                   moe4.OUT_BF16 | moe4.SF_MMA_LAYOUT, gws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    del wc, wsf, hc, hs
    h32 = oracle.bf16_to_f32(to_np(h, np.uint16))
    h_amax = np.abs(h32).max()
    sizes = np.diff(roffs)
    live = np.nonzero(sizes)[0]
    for e in [int(np.argmax(sizes)), int(live[0]), int(live[-1])]:
        lo, hi = int(roffs[e]), int(roffs[e + 1])
        rows = np.unique(np.concatenate([np.random.default_rng(e).choice(np.arange(lo, hi), 12), [lo, hi - 1]]))
        rhc, rhs, rhg = oracle.nvfp4_quantize(h32[rows], amax=h_amax)
        we = oracle.bf16_to_f32(to_np(w[e * d:(e + 1) * d], np.uint16))
        rwc, rws, rwg = oracle.nvfp4_quantize(we)
        Dref, S = oracle.grouped_gemm_m(oracle.nvfp4_dequantize(rhc, rhs, rhg),
                                        oracle.nvfp4_dequantize(rwc, rws, rwg)[None], np.array([0, len(rows)]))
        check_bf16(to_np(Y[torch.as_tensor(rows, device=DEV)], np.uint16), Dref, S)


def _swiglu_pair(xpc, xps, xg, wc, wsf, wg, offs, E, R, f, K, flags):
    """The fused gate/up GEMM + SwiGLU and, for comparison, the GEMM followed by moe4_swiglu_amax."""
    gws = moe4.workspace(moe4.moe4_workspace_size_gemm(0, R, E, 2 * f, K))
    gu_ref = torch.empty((R, 2 * f), dtype=torch.float32, device=DEV)
    moe4.grouped_expert_gemm_nvfp4(xpc, xps, xg, wc, wsf, wg, offs, E, R, 2 * f, K, gu_ref, moe4.OUT_F32 | flags, gws)
    h_ref = torch.empty((R, f), dtype=torch.int16, device=DEV)
    am_ref = torch.empty(1, dtype=torch.float32, device=DEV)
    moe4.moe4_swiglu_amax(gu_ref, R, f, h_ref, am_ref)
    gu = torch.full((R, 2 * f), float("nan"), dtype=torch.float32, device=DEV)
    h = torch.full((R, f), -1, dtype=torch.int16, device=DEV)
    am = torch.full((1,), 123.0, dtype=torch.float32, device=DEV)
    moe4.grouped_expert_gemm_nvfp4_swiglu(xpc, xps, xg, wc, wsf, wg, offs, E, R, f, K, gu, h, am, flags, gws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    return (gu, h, am), (gu_ref, h_ref, am_ref)


@pytest.mark.parametrize("sf_mma", [False, True])
def test_nvfp4_gate_up_with_swiglu_equals_gemm_then_swiglu(sf_mma):
    """grouped_expert_gemm_nvfp4_swiglu against the gate/up GEMM followed by moe4_swiglu_amax, bit
    for bit (GU, h and the amax of h): four experts (one empty), f = 256 (two tiles of 128 gate and
    128 up columns), both scale layouts."""
    sizes, f, K = [128, 256, 0, 384], 256, 512
    rng = np.random.default_rng(61)
    E, offs = len(sizes), _offs(sizes)
    R = int(offs[-1])
    a_bits = _bf16(rng, (R, K), t=True)
    b_bits = _bf16(rng, (E * 2 * f, K), 0.05)
    ac, asf, ag = nvfp4_quantize(to_dev(a_bits), 1, R, K)
    bc, bsf, bg = nvfp4_quantize(to_dev(b_bits), E, 2 * f, K)
    flags = 0
    if sf_mma:
        asf2, bsf2 = torch.empty_like(asf), torch.empty_like(bsf)
        moe4.moe4_sf_to_mma_layout(asf, 1, R, K // 16, asf2)
        moe4.moe4_sf_to_mma_layout(bsf, E, 2 * f, K // 16, bsf2)
        asf, bsf, flags = asf2, bsf2, moe4.SF_MMA_LAYOUT
    got, want = _swiglu_pair(ac, asf, ag, bc, bsf, bg, to_dev(offs), E, R, f, K, flags)
    for a, b, name in zip(got, want, ("GU", "h", "amax")):
        assert torch.equal(a, b), name
    # and the GEMM part against the oracle's float64 product
    rac, ras, rag = oracle.nvfp4_quantize(oracle.bf16_to_f32(a_bits))
    rbc, rbs, rbg = oracle.nvfp4_quantize(oracle.bf16_to_f32(b_bits).reshape(E, 2 * f, K))
    Dref, S = oracle.grouped_gemm_m(oracle.nvfp4_dequantize(rac, ras, rag), oracle.nvfp4_dequantize(rbc, rbs, rbg), offs)
    check_f32(to_np(got[0]), Dref, S, "fused GU")


def test_nvfp4_gate_up_with_swiglu_layer_shape():
    """The layer step's gate/up projection (16384 tokens x top-8 over 384 experts, 160k padded rows,
    d_model 4096, f = 2048, tile-layout scales): the fused GEMM + SwiGLU equals the GEMM followed
    by moe4_swiglu_amax, bit for bit, over the whole output."""
    T, d, f, E, k = 16384, 4096, 2048, 384, 8
    rng = np.random.default_rng(1)
    lg = (rng.standard_normal((T, E)) + rng.standard_normal(E)).astype(np.float32)
    idx, _ = oracle.route_topk(lg, k)
    rows_cap = T * k + 127 * E
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_of = torch.empty((T, k), dtype=torch.int32, device=DEV)
    src_of = torch.empty(rows_cap, dtype=torch.int32, device=DEV)
    moe4.moe4_permute_plan(to_dev(idx), T, k, E, offs, row_of, src_of, rows_cap,
                           moe4.workspace(moe4.moe4_workspace_size(moe4.OP_PERMUTE_PLAN, T, k, E)))
    torch.cuda.synchronize()
    Rp = int(to_np(offs)[-1])
    x = inputs.device_student_t((T, d), inputs.device_generator(22, 0, DEV), DEV).view(torch.int16)
    w = inputs.device_normal((E * 2 * f, d), 0.02, inputs.device_generator(22, 1, DEV), DEV).view(torch.int16)
    xc, xs, xg = nvfp4_quantize(x, 1, T, d)
    xpc, xps = empty_u8(Rp, d // 2), empty_u8(Rp, d // 16)
    moe4.moe4_permute_nvfp4(xc, xs, T, d, src_of, Rp, xpc, xps, moe4.SF_MMA_LAYOUT)
    del xc, xs, x
    wc, ws_, wg = nvfp4_quantize(w, E, 2 * f, d, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT)
    del w
    got, want = _swiglu_pair(xpc, xps, xg, wc, ws_, wg, offs, E, Rp, f, d, moe4.SF_MMA_LAYOUT)
    for a, b, name in zip(got, want, ("GU", "h", "amax")):
        assert torch.equal(a, b), name


def _swb_pair(aq, ae, bq, be, offs, E, M, f, K, gu, flags):
    """The fused dgrad + SwiGLU backward and the dgrad (binary32 dH) followed by moe4_swiglu_backward."""
    ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, E, f, K))
    dh = torch.empty((M, f), dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8(aq, ae, bq, be, offs, E, M, f, K, dh, moe4.OUT_F32 | moe4.GROUP_M | flags, ws)
    want = torch.empty((M, 2 * f), dtype=torch.int16, device=DEV)
    moe4.moe4_swiglu_backward(gu, dh, M, f, want)
    got = torch.full((M, 2 * f), -1, dtype=torch.int16, device=DEV)
    moe4.grouped_gemm_mxfp8_swiglu_backward(aq, ae, bq, be, offs, E, M, f, K, gu, got, flags, ws)
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    return got, want


@pytest.mark.parametrize("sf_mma", [False, True])
def test_mxfp8_dgrad_with_swiglu_backward_equals_unfused(sf_mma):
    """grouped_gemm_mxfp8_swiglu_backward against the rows-grouped dgrad (binary32 dH) followed by
    moe4_swiglu_backward, bit for bit: four experts (one empty), f = 512 (two 256-column tiles),
    K = 640, GU with values across the sigmoid's range."""
    rng = np.random.default_rng(71)
    sizes, f, K = [256, 0, 128, 384], 512, 640
    E, offs = len(sizes), _offs(sizes)
    M = int(offs[-1])
    a_bits = _bf16(rng, (M, K))
    b_bits = _bf16(rng, (E * f, K), 0.02)
    aq, ae = _mxfp8_rowwise(a_bits, M, K)
    bq, be = _mxfp8_rowwise(b_bits, E * f, K)
    flags = 0
    if sf_mma:
        ae2, be2 = torch.empty_like(ae), torch.empty_like(be)
        moe4.moe4_sf_to_mma_layout(ae, 1, M, K // 32, ae2)
        moe4.moe4_sf_to_mma_layout(be, 1, E * f, K // 32, be2)
        ae, be, flags = ae2, be2, moe4.SF_MMA_LAYOUT
    gu = to_dev((rng.standard_normal((M, 2 * f)) * 3).astype(np.float32))
    got, want = _swb_pair(aq, ae, bq, be, to_dev(offs), E, M, f, K, gu, flags)
    assert torch.equal(got, want), int((got != want).sum())


def test_mxfp8_dgrad_with_swiglu_backward_layer_shape():
    """The layer step's down-projection dgrad (160k padded rows over 384 experts of a top-8 plan,
    f = 2048, d_model 4096) with the SwiGLU backward: equal to the unfused pair over the whole dGU."""
    T, d, f, E, k = 16384, 4096, 2048, 384, 8
    rng = np.random.default_rng(2)
    lg = (rng.standard_normal((T, E)) + rng.standard_normal(E)).astype(np.float32)
    idx, _ = oracle.route_topk(lg, k)
    rows_cap = T * k + 127 * E
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_of = torch.empty((T, k), dtype=torch.int32, device=DEV)
    src_of = torch.empty(rows_cap, dtype=torch.int32, device=DEV)
    moe4.moe4_permute_plan(to_dev(idx), T, k, E, offs, row_of, src_of, rows_cap,
                           moe4.workspace(moe4.moe4_workspace_size(moe4.OP_PERMUTE_PLAN, T, k, E)))
    torch.cuda.synchronize()
    M = int(to_np(offs)[-1])
    dy = inputs.device_normal((M, d), 1.0, inputs.device_generator(23, 0, DEV), DEV).view(torch.int16)
    w = inputs.device_normal((E * f, d), 0.02, inputs.device_generator(23, 1, DEV), DEV).view(torch.int16)
    aq, ae = empty_u8(M, d), empty_u8(M, d // 32)
    moe4.mxfp8_quantize(dy, M, d, aq, ae, 0, 0, moe4.ROWWISE)
    bq, be = empty_u8(E * f, d), empty_u8(E * f, d // 32)
    moe4.mxfp8_quantize(w, E * f, d, bq, be, 0, 0, moe4.ROWWISE)
    del dy, w
    gu = inputs.device_normal((M, 2 * f), 2.0, inputs.device_generator(23, 2, DEV), DEV, dtype=torch.float32)
    got, want = _swb_pair(aq, ae, bq, be, offs, E, M, f, d, gu, 0)
    assert torch.equal(got, want), int((got != want).sum())
