"""Empty problems through every entry point: each returns MOE4_OK, writes nothing it has no rows
for, and still writes what the definition gives for an empty input (an empty tensor's global
decode scale 1, since amax = 0 gives g_enc = 1; an empty SwiGLU's amax 0; an empty dispatch
plan's zero offsets and all-padding source rows; a contraction with every group empty leaves the
FP32 masters unchanged, -lr * 0 = 0, and still reports their amax)."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_03_b300 import moe4
from gpu_helpers import DEV, to_np

pytestmark = pytest.mark.gpu
SENT = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    moe4.load()


def buf(n=4096):
    return torch.full((n,), SENT, dtype=torch.uint8, device=DEV)


def untouched(*bufs):
    torch.cuda.synchronize()
    return all(bool((b == SENT).all()) for b in bufs)


def f32(n, v=0.0):
    return torch.full((n,), v, dtype=torch.float32, device=DEV)


def test_quantisers_and_codecs_on_zero_rows():
    x, codes, sf, out = buf(), buf(), buf(), buf()
    ws = moe4.workspace(1024)
    g = f32(2, -3.0)
    moe4.nvfp4_quantize(x, 2, 0, 64, 64, codes, sf, g, None, moe4.FOUR_OVER_SIX, ws)
    assert untouched(codes, sf) and to_np(g).tolist() == [1.0, 1.0]
    g = f32(2, -3.0)
    moe4.nvfp4_quantize_f32(x, 2, 0, 64, 64, codes, sf, g, None, moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT, ws)
    assert untouched(codes, sf) and to_np(g).tolist() == [1.0, 1.0]
    moe4.nvfp4_dequantize(codes, sf, f32(1, 1.0), 1, 0, 64, out)
    moe4.mxfp8_requant_transpose_sr(codes, sf, f32(1, 1.0), 1, 0, 128, out, buf(), 1, 2, moe4.SR | moe4.SF_OUT_MMA)
    moe4.mxfp8_quantize(x, 0, 64, out, buf(), 0, 0, moe4.ROWWISE)
    moe4.mxfp8_quantize(x, 0, 64, out, buf(), 0, 0, moe4.COLWISE | moe4.SR)
    e = [buf() for _ in range(4)]
    moe4.mxfp8_quantize_rowcol(x, 0, 128, *e, flags=moe4.SF_OUT_MMA)
    assert untouched(out, *e)
    g = f32(1, -3.0)
    moe4.hadamard_quant(x, 0, 128, codes, sf, g, moe4.FOUR_OVER_SIX, ws)
    assert untouched(codes, sf) and to_np(g).tolist() == [1.0]
    moe4.hadamard_dequant(codes, sf, g, 0, 128, out)
    moe4.hadamard_quant(x, 0, 128, codes, sf, None, moe4.MXFP8)
    moe4.hadamard_dequant(codes, sf, None, 0, 128, out, moe4.MXFP8)
    assert untouched(codes, sf, out)
    # the weight path on matrices of no rows, whole and as its split, shared-SM passes on a slice
    q, e8, gw = buf(), buf(), buf(16)
    wf = moe4.FOUR_OVER_SIX | moe4.SR
    moe4.nvfp4_quantize_f32_requant(x, 2, 0, 64, f32(2, 1.0), codes, sf, gw, q, e8, 1, 3, None, wf)
    moe4.nvfp4_quantize_f32_requant(x, 2, 0, 64, f32(2, 1.0), codes, sf, gw, q, e8, 1, 3, None,
                                    wf | moe4.PASS_QUANT | moe4.SHARE_SMS, mat_base=5)
    moe4.nvfp4_quantize_f32_requant(x, 2, 0, 64, f32(2, 1.0), codes, sf, gw, q, e8, 1, 3, None,
                                    wf | moe4.PASS_REQUANT, mat_base=5)
    assert untouched(codes, sf, gw, q, e8)


def test_moe_steps_on_zero_tokens_and_rows():
    E, k = 8, 2
    offs = torch.full((E + 1,), 7, dtype=torch.int32, device=DEV)
    src_of = torch.zeros(127 * E, dtype=torch.int32, device=DEV)
    idx, w, row_of = buf(), buf(), buf()
    moe4.moe4_route_topk(buf(), 0, E, k, idx, w)
    moe4.moe4_permute_plan(idx, 0, k, E, offs, row_of, src_of, 127 * E,
                           moe4.workspace(moe4.moe4_workspace_size(moe4.OP_PERMUTE_PLAN, 0, k, E)))
    torch.cuda.synchronize()
    assert not bool(offs.any()) and bool((src_of == -1).all()) and untouched(idx, w, row_of)
    out = [buf() for _ in range(4)]
    moe4.moe4_permute_nvfp4(buf(), buf(), 0, 64, src_of, 0, out[0], out[1])
    moe4.moe4_swiglu(buf(), 0, 64, out[2])
    amax = f32(1, -1.0)
    moe4.moe4_swiglu_amax(buf(), 0, 64, out[3], amax)
    assert untouched(*out) and float(to_np(amax)[0]) == 0.0
    out = [buf() for _ in range(4)]
    moe4.moe4_swiglu_backward(buf(), buf(), 0, 64, out[0])
    moe4.moe4_swiglu_backward_mxfp8(buf(), buf(), 0, 64, *out)
    moe4.moe4_combine(buf(), row_of, w, 0, k, 64, out[1])
    moe4.moe4_combine_backward(buf(), row_of, w, src_of, 0, k, 64, 0, out[2])
    moe4.moe4_combine_backward_mxfp8(buf(), row_of, w, src_of, 0, k, 128, 0, *out, flags=moe4.SF_OUT_MMA)
    moe4.moe4_sgd_update(buf(), buf(), 0, 1e-3, out[3])
    assert untouched(*out)


def test_gemms_with_no_rows_or_no_contraction():
    E, N, K = 2, 256, 256
    offs0 = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    d = buf(1 << 16)
    ws = moe4.workspace(1 << 20)
    moe4.grouped_expert_gemm_nvfp4(buf(), buf(), f32(1, 1.0), buf(), buf(), f32(E, 1.0), offs0, E, 0, N, K, d,
                                   moe4.OUT_F32, ws)
    moe4.grouped_gemm_mxfp8(buf(), buf(), buf(), buf(), offs0, E, 0, N, K, d, moe4.OUT_F32 | moe4.GROUP_M, ws)
    assert untouched(d)
    # the gate/up GEMM with the SwiGLU and the down dgrad with its backward, on no rows: nothing
    # written but the amax of the empty h, 0
    h, dgu = buf(1 << 16), buf(1 << 16)
    hmax = f32(1, -1.0)
    moe4.grouped_expert_gemm_nvfp4_swiglu(buf(), buf(), f32(1, 1.0), buf(), buf(), f32(E, 1.0), offs0, E, 0, 128, K,
                                          d, h, hmax, 0, ws)
    moe4.grouped_gemm_mxfp8_swiglu_backward(buf(), buf(), buf(), buf(), offs0, E, 0, N, K, buf(), dgu, 0, ws)
    assert untouched(d, h, dgu) and float(to_np(hmax)[0]) == 0.0
    # every group empty along the contraction: D = 0
    M = 128
    dk = torch.full((E, M, N), 5.0, dtype=torch.float32, device=DEV)
    moe4.grouped_gemm_mxfp8(buf(), buf(), buf(), buf(), offs0, E, M, N, 0, dk, moe4.OUT_F32 | moe4.GROUP_K, ws)
    torch.cuda.synchronize()
    assert not bool(dk.any())
    # the fused SGD with an empty contraction: every expert is skipped, masters and amax untouched
    rng = np.random.default_rng(5)
    w0 = (rng.standard_normal((E, M, N)) * 0.02).astype(np.float32)
    w = torch.from_numpy(w0).to(DEV)
    amax = f32(E, -1.0)
    # operand buffers as large as the tensor maps describe ([M, 128] and [N, 128] bytes), though an
    # empty contraction loads none of them
    moe4.grouped_gemm_mxfp8_wgrad_sgd(buf(M * 128), buf(M * 4), buf(N * 128), buf(N * 4), offs0, E, M, N, 0, w, None,
                                      1e-3, amax, 0, ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(w), w0)
    assert np.all(to_np(amax) == -1.0)
