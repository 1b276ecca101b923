"""Pins of the oracle's support steps (routing, dispatch permutation, SwiGLU and its gradient,
combine and its gradient, SGD) and of its float64 reference GEMMs.

Routing follows the Inkling 2 Small model card (each token goes to 8 of 384 experts; "Thinking
Machines: Nvidia FP4 Up to 6x Faster, Runs Gain 8%", model-card update); dispatch is in NVFP4
("4-bit computation from the start of Inkling 2 Small's pretraining", communication paragraph).
The GEMM reference is checked against torch.matmul in float64 (a library routine).
"""
import numpy as np
import pytest
import torch


def test_topk_against_sorted_python(orc):
    rng = np.random.default_rng(0)
    T, E, k = 64, 24, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[3, :] = 0.5                     # all tied: lowest indices win
    logits[7, 5] = logits[7, 2] = 9.0      # tie between two top experts
    idx, w = orc.route_topk(logits, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        assert list(idx[t]) == order
        sel = np.array([float(logits[t, e]) for e in order])
        ex = np.exp(sel - sel.max())
        assert np.allclose(w[t], ex / ex.sum(), rtol=1e-6)
    assert list(idx[3]) == [0, 1, 2, 3]
    assert list(idx[7][:2]) == [2, 5]
    assert np.allclose(w.sum(axis=1), 1.0, rtol=1e-6)


def test_permute_plan_and_rows(orc):
    rng = np.random.default_rng(1)
    T, E, k = 300, 16, 3
    logits = rng.standard_normal((T, E)).astype(np.float32) + rng.standard_normal(E).astype(np.float32) * 2
    idx, w = orc.route_topk(logits, k)
    offs, row_of = orc.permute_plan(idx, E)
    counts = np.bincount(idx.reshape(-1), minlength=E)
    assert offs[0] == 0 and np.all(np.diff(offs) % 128 == 0)
    assert np.all(np.diff(offs) >= counts) and np.all(np.diff(offs) < counts + 128)
    flat = row_of.reshape(-1)
    assert len(set(flat.tolist())) == flat.size
    for e in range(E):
        members = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        rows = [int(row_of[t, j]) for t, j in members]
        assert rows == list(range(offs[e], offs[e] + len(members)))   # stable in (token, slot)
    src = rng.integers(0, 256, (T, 8)).astype(np.uint8)
    g = orc.permute_rows(src, row_of, int(offs[-1]))
    used = np.zeros(int(offs[-1]), bool)
    used[flat] = True
    assert np.all(g[~used] == 0)
    for t in range(T):
        for j in range(k):
            assert np.array_equal(g[row_of[t, j]], src[t])


def test_combine_against_loop(orc):
    rng = np.random.default_rng(2)
    T, k, d, R = 5, 3, 16, 40
    yh = orc.f32_to_bf16(rng.standard_normal((R, d)).astype(np.float32))
    row_of = rng.permutation(R)[:T * k].reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    got = orc.bf16_to_f32(orc.combine(yh, row_of, w))
    yf = orc.bf16_to_f32(yh)
    for t in range(T):
        for c in range(d):
            acc = np.float32(0.0)
            for j in range(k):
                acc = np.float32(acc + np.float32(w[t, j] * yf[row_of[t, j], c]))
            want = torch.tensor([float(acc)], dtype=torch.float32).to(torch.bfloat16).float().item()
            assert got[t, c] == want


def test_swiglu_special_points(orc):
    gu = np.array([[0.0, 3.0, 2.0, 5.0],      # g = (0, 3), u = (2, 5)
                   [40.0, -40.0, 1.5, 7.0]], np.float32)
    h = orc.swiglu(gu)
    assert h[0, 0] == 0.0
    assert np.isclose(h[0, 1], 3.0 / (1 + np.exp(-3.0)) * 5.0, rtol=1e-7)
    assert np.isclose(h[1, 0], 40.0 * 1.5, rtol=1e-7)
    assert abs(h[1, 1]) < 2e-15  # silu(-40) * 7 = -40 e^-40 * 7


def test_sgd_update_exact(orc):
    w = np.float32([1.0, -2.0, 3.5])
    dw = np.float32([0.5, 0.25, -4.0])
    w2, wb = orc.sgd_update(w, dw, 0.5)
    assert list(w2) == [0.75, -2.125, 5.5]
    assert list(orc.bf16_to_f32(wb)) == [0.75, -2.125, 5.5]


def test_grouped_gemm_m_against_torch(orc):
    rng = np.random.default_rng(3)
    E, N, K = 4, 24, 64
    offs = np.array([0, 128, 128, 384, 512], np.int32)   # expert 1 is empty
    A = rng.standard_normal((512, K)).astype(np.float32)
    B = rng.standard_normal((E, N, K)).astype(np.float32)
    D, S = orc.grouped_gemm_m(A, B, offs)
    for e in range(E):
        lo, hi = offs[e], offs[e + 1]
        ref = torch.from_numpy(A[lo:hi]).double() @ torch.from_numpy(B[e]).double().T
        assert np.allclose(D[lo:hi], ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(S >= np.abs(D) - 1e-9)


def test_grouped_gemm_k_against_torch(orc):
    rng = np.random.default_rng(4)
    M, N, R = 16, 8, 384
    offs = np.array([0, 256, 256, 384], np.int32)
    A = rng.standard_normal((M, R)).astype(np.float32)
    B = rng.standard_normal((N, R)).astype(np.float32)
    D, S = orc.grouped_gemm_k(A, B, offs)
    assert np.all(D[1] == 0)
    for e in (0, 2):
        lo, hi = offs[e], offs[e + 1]
        ref = torch.from_numpy(A[:, lo:hi]).double() @ torch.from_numpy(B[:, lo:hi]).double().T
        assert np.allclose(D[e], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_swiglu_backward_against_autograd(orc):
    # torch's autograd differentiates silu(g) * u in float64 on its own (a library routine): a
    # dropped term, a sign or the gate/up halves swapped in the oracle's closed form fails here
    rng = np.random.default_rng(11)
    rows, f = 6, 24
    gu = (rng.standard_normal((rows, 2 * f)) * 3).astype(np.float32)
    gu[0, :4] = [0.0, -30.0, 30.0, 1e-3]
    dh = rng.standard_normal((rows, f)).astype(np.float32)
    g = torch.from_numpy(gu[:, :f]).double().requires_grad_(True)
    u = torch.from_numpy(gu[:, f:]).double().requires_grad_(True)
    (torch.nn.functional.silu(g) * u).backward(torch.from_numpy(dh).double())
    want = torch.cat([g.grad, u.grad], dim=1).numpy()
    got = orc.swiglu_backward(gu, dh)
    assert got.shape == (rows, 2 * f) and got.dtype == np.float32
    assert np.allclose(got.astype(np.float64), want, rtol=2e-7, atol=1e-30)


def test_swiglu_forward_against_torch_silu(orc):
    rng = np.random.default_rng(12)
    gu = (rng.standard_normal((5, 32)) * 4).astype(np.float32)
    g, u = torch.from_numpy(gu[:, :16]).double(), torch.from_numpy(gu[:, 16:]).double()
    want = (torch.nn.functional.silu(g) * u).numpy()
    assert np.allclose(orc.swiglu(gu), want, rtol=2e-7, atol=1e-30)


def test_combine_backward_is_the_adjoint_of_the_combine(orc):
    # <combine(yhat), dy> = <yhat, combine_backward(dy)>.  Small integers and power-of-two
    # weights keep every product, sum and bf16 rounding exact, so the identity holds exactly;
    # a transposed index (token for row) or a weight taken from the wrong slot breaks it
    rng = np.random.default_rng(13)
    T, k, d, R = 40, 4, 32, 200
    row_of = rng.permutation(R)[:T * k].reshape(T, k).astype(np.int32)
    w = rng.choice(np.float32([1.0, 0.5, 0.25]), size=(T, k)).astype(np.float32)
    yh = orc.f32_to_bf16(rng.integers(-4, 5, (R, d)).astype(np.float32))
    dy = orc.f32_to_bf16(rng.integers(-4, 5, (T, d)).astype(np.float32))
    y = orc.bf16_to_f32(orc.combine(yh, row_of, w)).astype(np.float64)
    dyhat = orc.bf16_to_f32(orc.combine_backward(dy, row_of, w, R)).astype(np.float64)
    lhs = float(np.sum(y * orc.bf16_to_f32(dy)))
    rhs = float(np.sum(orc.bf16_to_f32(yh).astype(np.float64) * dyhat))
    assert lhs == rhs and lhs != 0.0
    # rows no (token, slot) maps to are zero
    unused = np.setdiff1d(np.arange(R), row_of.reshape(-1))
    assert unused.size == R - T * k and np.all(dyhat[unused] == 0)


def test_dispatch_backward_is_the_adjoint_of_the_gather(orc):
    # <gather(x), g> = <x, dispatch_backward(g)> with gather(x)[row_of[t, j]] = x[t]: small integers
    # keep every sum and bf16 rounding exact, so the identity holds exactly; a transposed index or
    # a dropped slot breaks it
    rng = np.random.default_rng(14)
    T, k, d, R = 30, 8, 16, 400
    row_of = rng.permutation(R)[:T * k].reshape(T, k).astype(np.int32)
    x = rng.integers(-4, 5, (T, d)).astype(np.float32)
    g = orc.f32_to_bf16(rng.integers(-4, 5, (R, d)).astype(np.float32))
    xp = orc.permute_rows(x, row_of, R).astype(np.float64)
    dx = orc.bf16_to_f32(orc.dispatch_backward(g, row_of)).astype(np.float64)
    lhs = float(np.sum(xp * orc.bf16_to_f32(g)))
    rhs = float(np.sum(x.astype(np.float64) * dx))
    assert lhs == rhs and lhs != 0.0
    # one slot: the gradient row itself; slot order matters only through rounding
    one = orc.dispatch_backward(g, row_of[:, :1])
    assert np.array_equal(one, g[row_of[:, 0]])
