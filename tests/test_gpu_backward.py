"""GPU parity of the backward pass (dQ, dK, dV by recomputation from LSE)
against the fp64 backward oracle, on the same bf16 inputs.

Bar, derived from bf16's unit roundoff u = 2^-8 (P and dS are rounded to bf16
as MMA operands, D uses the forward's bf16 O, outputs are bf16): for each
gradient G, max|err| <= 2e-2 * max|G_ref| (about 5u) and mean|err| <=
5e-3 * mean|G_ref| (about 1.3u). At full size, where the fp64 oracle is too
slow, two identities that hold at any size are checked instead:
sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i over each head.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import WORKLOADS, custom, make_qkv

pytestmark = pytest.mark.gpu


def upstream(q, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(q.shape, generator=g).to(torch.bfloat16)


def run_fwd_bwd(q, k, v, do, causal, scale, own_ws=True):
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, Sq), device="cuda")
    _capi.check(_capi.fa_prefill_forward(qd, kd, vd, o, lse, B, H, Sq, Sk, d, causal, scale), "fwd")
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    ws, nb = None, 0
    if own_ws:
        nb = _capi.fa_backward_workspace_size(B, H, Sq, Sk, d)
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    _capi.check(_capi.fa_backward(qd, kd, vd, o, lse, dod, dq, dk, dv, B, H, Sq, Sk, d, causal,
                                  scale, ws, nb), "fa_backward")
    torch.cuda.synchronize()
    _capi.check(_capi.fa_device_status(), "device status")
    return dq.double().cpu().numpy(), dk.double().cpu().numpy(), dv.double().cpu().numpy()


def check_grad(name, got, ref):
    assert np.all(np.isfinite(got)), f"{name}: non-finite"
    err = np.abs(got - ref)
    scale_max, scale_mean = np.max(np.abs(ref)), np.mean(np.abs(ref))
    assert err.max() <= 2e-2 * scale_max + 1e-4, (name, err.max(), scale_max)
    assert err.mean() <= 5e-3 * scale_mean + 1e-5, (name, err.mean(), scale_mean)


CASES = [
    # B, H, Sq, Sk, d, causal
    (1, 2, 256, 256, 128, True),
    (1, 2, 300, 300, 128, True),
    (2, 1, 129, 129, 64, True),
    (1, 2, 384, 384, 128, False),
    (1, 1, 200, 500, 128, True),    # bottom-right: Sq < Sk
    (1, 1, 300, 100, 64, True),     # Sq > Sk: rows with no visible key
    (1, 2, 17, 33, 128, False),
    (1, 1, 1000, 1000, 128, True),
    (1, 2, 700, 700, 64, True),     # d = 64: the key and value rings wrap
    (1, 1, 640, 1100, 64, False),   # 9 key tiles, non-causal
    (2, 1, 257, 900, 128, True),    # Sq < Sk, ragged query and key tails
]


def test_backward_rows_without_keys_after_cold_cache():
    """Query tiles that see no key get dQ = 0. They load nothing: a Q load still
    landing in the buffer that stages their zero tile would overwrite it. L2 is
    flushed before each run so that such a load would be slow."""
    B, H, Sq, Sk, d = 1, 2, 300, 100, 64
    w = custom(B, H, Sq, Sk, d, True, seed=Sq + 3 * Sk, q_factor=2.0)
    q, k, v = make_qkv(w)
    do = upstream(q, w.seed)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, True, w.scale)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(5):
        flush.fill_(1)
        dq, dk, dv = run_fwd_bwd(q, k, v, do, True, w.scale)
        assert np.all(dq[:, :, :Sq - Sk] == 0.0)  # rows 0 .. Sq-Sk-1 see no key
        check_grad("dq", dq, rq)
        check_grad("dk", dk, rk)
        check_grad("dv", dv, rv)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
def test_backward_matches_oracle(case):
    B, H, Sq, Sk, d, causal = case
    w = custom(B, H, Sq, Sk, d, causal, seed=Sq + 3 * Sk, q_factor=2.0)
    q, k, v = make_qkv(w)
    do = upstream(q, w.seed)
    dq, dk, dv = run_fwd_bwd(q, k, v, do, causal, w.scale, own_ws=Sq % 2 == 0)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, causal, w.scale)
    check_grad("dq", dq, rq)
    check_grad("dk", dk, rk)
    check_grad("dv", dv, rv)


def test_backward_2k_workload_one_batch():
    """The 2K prefill workload's first batch element, every gradient element."""
    w = WORKLOADS["prefill_b4h32s2048d128_causal"]
    q, k, v = make_qkv(w)
    q, k, v = q[:1, :4].contiguous(), k[:1, :4].contiguous(), v[:1, :4].contiguous()
    do = upstream(q, 5)
    dq, dk, dv = run_fwd_bwd(q, k, v, do, True, w.scale)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, True, w.scale)
    check_grad("dq", dq, rq)
    check_grad("dk", dk, rk)
    check_grad("dv", dv, rv)


def test_backward_headline_shape_sampled_rows():
    """B=4, H=32, S=8192, d=128 causal, in the configuration the benchmark times: dQ of
    sampled query rows and dK, dV of sampled key rows of two heads, each against the
    oracle's per-row backward (same bar, taken over the sampled rows)."""
    w = WORKLOADS["prefill_b4h32s8192d128_causal"]
    q, k, v = make_qkv(w)
    do = upstream(q, 11)
    dq, dk, dv = run_fwd_bwd(q, k, v, do, True, w.scale)
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
    g = np.random.default_rng(3)
    rows = sorted(set([0, 127, 128, 4095, 8191] + g.integers(0, 8192, 27).tolist()))
    for b, h in ((0, 0), (3, 31)):
        rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, True, w.scale, b, h, rows, rows)
        check_grad("dq", dq[b, h, rows], rq)
        check_grad("dk", dk[b, h, rows], rk)
        check_grad("dv", dv[b, h, rows], rv)


def test_backward_is_deterministic():
    """No atomics: two runs give the same bits."""
    w = custom(1, 2, 520, 520, 128, True, seed=21, q_factor=2.0)
    q, k, v = make_qkv(w)
    do = upstream(q, 22)
    a = run_fwd_bwd(q, k, v, do, True, w.scale)
    b = run_fwd_bwd(q, k, v, do, True, w.scale)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_backward_cuda_graph_replay():
    """The backward (three kernels, the last launched with programmatic stream
    serialization) captured in a CUDA graph and replayed on new inputs gives the
    bits an eager call gives, and the graph's completion orders a dependent copy."""
    w = custom(1, 2, 640, 640, 128, True, seed=31, q_factor=2.0)
    q, k, v = (t.cuda() for t in make_qkv(w))
    do = upstream(q.cpu(), 32).cuda()
    B, H, Sq, Sk, d = w.B, w.H, w.Sq, w.Sk, w.d
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nb = _capi.fa_backward_workspace_size(B, H, Sq, Sk, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def fwd_bwd(stream):
        _capi.check(_capi.fa_prefill_forward(q, k, v, o, lse, B, H, Sq, Sk, d, True, w.scale,
                                             stream), "fwd")
        _capi.check(_capi.fa_backward(q, k, v, o, lse, do, dq, dk, dv, B, H, Sq, Sk, d, True,
                                      w.scale, ws, nb, stream), "bwd")

    with torch.cuda.stream(s):  # warm-up (kernel attributes) before capture
        fwd_bwd(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fwd_bwd(s)
        dk_copy = dk.clone()  # ordered after the whole backward
    for seed in (33, 34):
        qn, kn, vn = make_qkv(custom(B, H, Sq, Sk, d, True, seed=seed, q_factor=2.0))
        q.copy_(qn); k.copy_(kn); v.copy_(vn)
        g.replay()
        torch.cuda.synchronize()
        got = (dq.clone(), dk.clone(), dv.clone(), dk_copy.clone())
        with torch.cuda.stream(s):
            fwd_bwd(s)
        torch.cuda.synchronize()
        assert torch.equal(got[0], dq) and torch.equal(got[1], dk) and torch.equal(got[2], dv)
        assert torch.equal(got[3], dk)


PEAKED = [
    # B, H, Sq, Sk, d, causal: Q x 4 (a few keys dominate each row) with few keys
    (1, 2, 5, 7, 128, True),
    (1, 1, 2, 7, 64, False),
    (1, 3, 1, 64, 64, True),
]


@pytest.mark.parametrize("case", PEAKED, ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
def test_backward_peaked_rows_within_the_output_rounding_bound(case):
    """D_i = dO_i . O_i uses the forward's output, which is bf16. Where one key
    dominates a row, dP_ij - D_i cancels and the rounding of O (at most 2^-9 of
    each |O_id|) shows in dS and so in dQ and dK beyond the general bar. Against
    the exact gradient the error stays within the general bar plus the bound
    that rounding propagates:
        |dD_i| <= 2^-9 sum_d |dO_id O_id|,
        |d dQ_i| <= scale |dD_i| sum_j P_ij |K_j|,  |d dK_j| <= scale sum_i P_ij |dD_i| |Q_i|,
    and dV (no D) stays within the general bar."""
    B, H, Sq, Sk, d, causal = case
    w = custom(B, H, Sq, Sk, d, causal, seed=1, q_factor=4.0)
    q, k, v = make_qkv(w)
    do = upstream(q, 1)
    dq, dk, dv = run_fwd_bwd(q, k, v, do, causal, w.scale)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, causal, w.scale)
    ro, _ = oracle.attention(q, k, v, causal, w.scale)
    qn, kn, dn = q.double().numpy(), k.double().numpy(), do.double().numpy()
    scale = float(np.float32(w.scale))
    bq, bk = np.zeros_like(rq), np.zeros_like(rk)
    for b in range(B):
        for h in range(H):
            P = np.stack([oracle.probs_row(q, k, causal, w.scale, b, h, i) for i in range(Sq)])
            dD = 2.0 ** -9 * np.abs(dn[b, h] * ro[b, h]).sum(-1)          # [Sq]
            bq[b, h] = scale * dD[:, None] * (P @ np.abs(kn[b, h]))
            bk[b, h] = scale * (P * dD[:, None]).T @ np.abs(qn[b, h])
    for name, got, ref, bound in (("dq", dq, rq, bq), ("dk", dk, rk, bk)):
        err = np.abs(got - ref)
        assert np.all(err <= 2e-2 * np.abs(ref).max() + 1.01 * bound + 1e-4), \
            (name, float((err - bound).max()), float(np.abs(ref).max()))
    check_grad("dv", dv, rv)
