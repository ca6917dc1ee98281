"""Pins for the fp64 backward oracle (gradients of the attention definition).

Checked against torch's fp64 autograd through scaled_dot_product_attention
(a library routine), central finite differences of the independent numpy
forward, and closed forms (a constant V makes O independent of Q and K; one
key makes O equal to its value row).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.numpy_ref import attention_np, to_f64
from exact_tiled_attention_03_gb300.inputs import custom, make_qkv

TOL = 1e-11


def case(B, H, Sq, Sk, d, causal, seed=0, factor=1.0):
    w = custom(B, H, Sq, Sk, d, causal, seed=seed, q_factor=factor)
    q, k, v = make_qkv(w)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    return w, q, k, v, do


SHAPES = [(1, 2, 7, 7, 16, True), (2, 1, 5, 13, 8, True), (1, 1, 9, 4, 8, True),
          (1, 2, 6, 11, 16, False), (1, 1, 33, 40, 32, True)]


@pytest.mark.parametrize("shape", SHAPES)
def test_matches_torch_autograd_fp64(shape):
    w, q, k, v, do = case(*shape, seed=61, factor=2.0)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, w.causal, w.scale)
    qd, kd, vd = (t.double().requires_grad_() for t in (q, k, v))
    mask = None
    if w.causal:
        i = torch.arange(w.Sq)[:, None]
        j = torch.arange(w.Sk)[None, :]
        mask = j <= i + (w.Sk - w.Sq)
    sc = float(np.float32(w.scale))
    o = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=sc)
    if mask is not None:   # rows with no visible key: torch gives NaN, the definition gives 0
        empty = ~mask.any(dim=-1)
        o = o.masked_fill(empty[None, None, :, None], 0.0)
    o.backward(do.double())
    for mine, ref in ((dq, qd.grad), (dk, kd.grad), (dv, vd.grad)):
        ref = torch.nan_to_num(ref, nan=0.0).numpy()
        assert np.max(np.abs(mine - ref)) < TOL * max(1.0, np.max(np.abs(ref)))


def test_matches_central_finite_differences_of_the_numpy_forward():
    """dL/dx for L = sum(dO * O), O from the independent numpy forward, at a few entries."""
    w, q, k, v, do = case(1, 1, 6, 9, 8, True, seed=67, factor=2.0)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, True, w.scale)
    Q, K, V, G = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    sc = float(np.float32(w.scale))
    loss = lambda Q_, K_, V_: float(np.sum(G * attention_np(Q_, K_, V_, True, sc)[0]))
    h = 1e-6
    rng = np.random.default_rng(0)
    for name, X, grad in (("q", Q, dq), ("k", K, dk), ("v", V, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"q": (Xp, K, V), "k": (Q, Xp, V), "v": (Q, K, Xp)}[name]
            args_m = {"q": (Xm, K, V), "k": (Q, Xm, V), "v": (Q, K, Xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) < 1e-6 * max(1.0, abs(fd)), (name, idx)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_zero_query_and_key_gradients(causal):
    """With every value row equal, O does not depend on Q or K; sum_j dV_j = sum_i dO_i."""
    w, q, k, v, do = case(2, 2, 9, 9, 16, causal, seed=71, factor=3.0)
    v = torch.full_like(v, 0.75)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, w.scale)
    assert np.max(np.abs(dq)) < 1e-13 and np.max(np.abs(dk)) < 1e-13
    assert np.max(np.abs(dv.sum(axis=2) - to_f64(do).sum(axis=2))) < 1e-12


def test_single_key_routes_all_gradient_to_its_value():
    w, q, k, v, do = case(1, 3, 5, 1, 8, False, seed=73)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, False, w.scale)
    assert np.max(np.abs(dq)) == 0.0 and np.max(np.abs(dk)) == 0.0
    assert np.max(np.abs(dv[:, :, 0] - to_f64(do).sum(axis=2))) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_the_full_backward(causal):
    """The row-subset backward agrees with the full one (different loop order, same math)."""
    w, q, k, v, do = case(2, 3, 70, 90, 16, causal, seed=79, factor=2.0)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, w.scale)
    qrows, krows = [0, 5, 69, 33], [0, 1, 89, 40, 22]
    for b, h in ((0, 0), (1, 2)):
        rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, causal, w.scale, b, h, qrows, krows)
        assert np.max(np.abs(rq - dq[b, h, qrows])) < TOL
        assert np.max(np.abs(rk - dk[b, h, krows])) < TOL
        assert np.max(np.abs(rv - dv[b, h, krows])) < TOL
