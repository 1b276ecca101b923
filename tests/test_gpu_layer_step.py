"""The layer step's orchestration at full size (bench.py's LayerStep: 16384 tokens, 384 experts,
top-8, d_model 4096, SwiGLU width 2048): the weight path as the step runs it (four expert chunks
per projection on two streams, each chunk's quantiser on part of each SM beside the previous
chunk's requantiser, every call on slices with its matrix base) writes, for every expert that
received rows, exactly the bytes of one call over the whole stack; experts without rows are
skipped by both."""
import os
import sys

import numpy as np
import pytest
import torch

from precision_moe_numerics_03_b300 import moe4
from gpu_helpers import DEV, to_np

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_layer_step_weight_path_equals_one_call_per_projection():
    sys.path.insert(0, ROOT)
    import bench
    moe4.load()
    T, d, f, E, k = 16384, 4096, 2048, 384, 8
    s = bench.LayerStep(T, d, f, E, k, DEV)
    s.m.moe4_route_topk(s.logits, T, E, k, s.idx, s.w)
    s.m.moe4_permute_plan(s.idx, T, k, E, s.offs, s.row_of, s.src_of, s.rows_cap, s.plan_ws)
    seed = 4321
    s.weight_path(seed, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert moe4.moe4_get_status() == moe4.OK
    live = np.nonzero(np.diff(to_np(s.offs)))[0]
    assert 0 < len(live) < E  # the routing leaves some experts empty: the skip path is exercised
    wf = moe4.FOUR_OVER_SIX | moe4.SR | moe4.SF_MMA_LAYOUT | moe4.SF_OUT_MMA
    for W, am, got, rows, cols, sid in (
            (s.W32_gu, s.amax_gu, (s.Wgu_c, s.Wgu_s, s.Wgu_g, s.WguT_q, s.WguT_e), 2 * f, d, 3),
            (s.W32_d, s.amax_d, (s.Wd_c, s.Wd_s, s.Wd_g, s.WdT_q, s.WdT_e), d, f, 1)):
        ref = [torch.empty_like(t) for t in got]
        moe4.nvfp4_quantize_f32_requant(W, E, rows, cols, am, *ref, seed, sid, s.offs, wf)
        torch.cuda.synchronize()
        idx = torch.as_tensor(live, device=DEV)
        for a, b in zip(got, ref):
            assert torch.equal(a.index_select(0, idx), b.index_select(0, idx))
        del ref
