"""GPU parity at scale 0 and at negative scales, on every kernel, against the
unchanged fp64 oracle.

The pages make the softmax scale a plain factor of the scores (S = Q K^T / sqrt(d)
in "Warmup Guide", Chapter 4; none at all in the Mechanics pseudocode of
"FlashAttention, speculative decoding, quantisation and parallelism"), so every
finite value is valid. Scale 0 gives uniform weights over the visible keys (the
oracle's pinned closed form: O = mean of the visible V rows, LSE = ln of their
count); a negative scale turns the row max into the min of the raw scores, which
the kernels handle by forming -Q K^T on the tensor cores (the tcgen05 operand
negation, or -Q in the mma.sync verify kernel) and running the softmax with
|scale|. Q x 4 makes the reference move often, so the lazy-rescale path runs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import custom, make_paged_kv, make_qkv, make_qkv_fp8, make_tree_masks
from parity import compare, oracle_full, run
from test_gpu_backward import check_grad, run_fwd_bwd, upstream
from test_gpu_fp8 import run_fp8
from test_gpu_verify_ext import dense_visible, run_paged, run_verify_tree

pytestmark = pytest.mark.gpu

MULTS = [0.0, -1.0, -2.0]  # times 1/sqrt(d)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _capi.load()


def ids(c):
    return "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else "n")


PREFILL = [
    # B, H, Sq, Sk, d, causal
    (1, 2, 300, 300, 128, True),
    (1, 2, 384, 640, 128, False),
    (1, 1, 200, 520, 128, True),     # Sq < Sk: bottom-right offset
    (1, 2, 300, 100, 64, True),      # Sk < Sq: rows with no visible key
    (2, 1, 257, 257, 64, False),
]


@pytest.mark.parametrize("mult", MULTS)
@pytest.mark.parametrize("case", PREFILL, ids=ids)
def test_prefill_any_finite_scale(case, mult):
    B, H, Sq, Sk, d, causal = case
    w = custom(B, H, Sq, Sk, d, causal, seed=Sq + Sk + d, q_factor=4.0)
    q, k, v = make_qkv(w)
    scale = mult / math.sqrt(d)
    o, lse = run("fa_prefill_forward", q, k, v, causal, scale)
    ro, rl = oracle_full(q, k, v, causal, scale)
    compare(o, lse, ro, rl)


def test_prefill_negative_scale_is_the_negated_query_bit_for_bit():
    """scale -c on Q runs the same arithmetic as +c on -Q (the MMA negates exactly)."""
    w = custom(1, 2, 640, 640, 128, True, seed=5, q_factor=2.0)
    q, k, v = make_qkv(w)
    a = run("fa_prefill_forward", q, k, v, True, -w.scale)
    b = run("fa_prefill_forward", -q, k, v, True, w.scale)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("mult", MULTS)
@pytest.mark.parametrize("n_split", [1, 3])
@pytest.mark.parametrize("case", [(2, 4, 5, 1000, 128, True), (1, 3, 16, 700, 64, False),
                                  (2, 2, 8, 6, 128, True)], ids=ids)
def test_verify_any_finite_scale(case, n_split, mult):
    B, H, Sq, Sk, d, causal = case
    if n_split > -(-Sk // 64):
        pytest.skip("more splits than 64-key chunks")
    w = custom(B, H, Sq, Sk, d, causal, seed=Sq * 7 + Sk, q_factor=4.0)
    q, k, v = make_qkv(w)
    scale = mult / math.sqrt(d)
    o, lse = run("fa_verify_forward", q, k, v, causal, scale, n_split=n_split)
    ro, rl = oracle_full(q, k, v, causal, scale)
    compare(o, lse, ro, rl)


@pytest.mark.parametrize("mult", [0.0, -1.0])
def test_main_entry_point_any_finite_scale(mult):
    """fa_forward on both of its paths (split-KV for Sq <= 16, prefill otherwise)."""
    for (Sq, Sk) in ((5, 900), (256, 256)):
        w = custom(1, 2, Sq, Sk, 128, True, seed=Sq + 1, q_factor=2.0)
        q, k, v = make_qkv(w)
        scale = mult * w.scale
        o, lse = run("fa_forward", q, k, v, True, scale)
        ro, rl = oracle_full(q, k, v, True, scale)
        compare(o, lse, ro, rl)


@pytest.mark.parametrize("mult", [0.0, -1.0])
def test_verify_tree_any_finite_scale(mult):
    B, H, Sq, Sk, d = 2, 3, 5, 300, 128
    w = custom(B, H, Sq, Sk, d, True, seed=99, q_factor=2.0)
    q, k, v = make_qkv(w)
    masks = make_tree_masks(B, Sq, seed=Sk)
    scale = mult * w.scale
    o, lse = run_verify_tree(q, k, v, masks, scale, 3)
    ro, rl = oracle.attention_masked(q, k, v, dense_visible(masks.numpy(), Sq, [Sk] * B), scale)
    compare(o, lse, ro, rl)


@pytest.mark.parametrize("mult", [0.0, -1.0])
@pytest.mark.parametrize("page_size", [16, 64])
def test_verify_paged_any_finite_scale(page_size, mult):
    """Paged K/V through a block table; each sequence against the oracle on its
    logical K/V."""
    B, H, Sq, d, Smax = 3, 2, 5, 128, 700
    lens = [700, 69, 333]
    w = custom(B, H, Sq, Smax, d, True, seed=page_size + 3, q_factor=2.0)
    q, k, v = make_qkv(w)
    kp, vp, table, lens_t = make_paged_kv(k, v, lens, page_size, seed=page_size)
    scale = mult * w.scale
    o, lse = run_paged(q, kp, vp, table, lens_t, page_size, Smax, True, None, scale, 3)
    for b in range(B):
        Sk = lens[b]
        ro, rl = oracle.attention(q[b:b + 1], k[b:b + 1, :, :Sk], v[b:b + 1, :, :Sk], True, scale)
        compare(o[b:b + 1], lse[b:b + 1], ro, rl)


@pytest.mark.parametrize("mult", MULTS)
@pytest.mark.parametrize("case", [(1, 2, 300, 300, 128, True), (1, 1, 200, 500, 128, True),
                                  (1, 2, 384, 384, 64, False)], ids=ids)
def test_backward_any_finite_scale(case, mult):
    """dK and dQ carry the signed scale; P is rebuilt with |scale| from -Q K^T."""
    B, H, Sq, Sk, d, causal = case
    w = custom(B, H, Sq, Sk, d, causal, seed=Sq + 5 * Sk, q_factor=2.0)
    q, k, v = make_qkv(w)
    do = upstream(q, w.seed)
    scale = mult / math.sqrt(d)
    dq, dk, dv = run_fwd_bwd(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, causal, scale)
    check_grad("dq", dq, rq)
    check_grad("dk", dk, rk)
    check_grad("dv", dv, rv)


@pytest.mark.parametrize("mult", MULTS)
@pytest.mark.parametrize("case", [(1, 2, 300, 300, True), (1, 2, 520, 200, True),
                                  (1, 1, 384, 700, False)],
                         ids=lambda c: "b{}h{}q{}k{}{}".format(*c[:4], "c" if c[4] else "n"))
def test_fp8_any_finite_scale(case, mult):
    B, H, Sq, Sk, causal = case
    w = custom(B, H, Sq, Sk, 128, causal, seed=Sq * 3 + Sk, q_factor=2.0)
    q8, k8, v8, ds = make_qkv_fp8(w)
    scale = mult * w.scale
    o, lse = run_fp8(q8, k8, v8, causal, scale, ds)
    o_ref, lse_ref = oracle.attention_fp8(q8, k8, v8, causal, scale, ds)
    compare(o, lse, o_ref, lse_ref)
