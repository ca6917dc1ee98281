"""GPU parity of the FP8 forward (fa_forward_fp8), through the C ABI, against the
oracle's FP8 path on the same seeded E4M3 inputs, element by element.

The oracle rounds P to E4M3 at the scale 2^7 against the row's power-of-two
max. The kernel's scale is 2^4 to 2^9 against its trailing reference, which
gives the same weights (up to an exact power of two) for every weight of at
least 2^-10 of the row max; smaller weights may round on E4M3's subnormal
grid. The other differences are fp32 accumulation, the exp2 approximation
(which can move a weight that sits within ~1e-7 of an E4M3 rounding tie to the
neighbouring grid point) and the bf16 output. The bar
is the one of the bf16 path: O max-abs 2e-2, mean-abs 2e-3, LSE 1e-3. One case
also checks the kernel against the unrounded definition with the bound
E4M3's three mantissa bits give.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import WORKLOADS, HEADLINE, custom, make_qkv_fp8, sample_rows
from parity import alloc_outputs, check_guard, compare, gather_rows, views

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _capi.load()


def u8(t):
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


# ---------------------------------------------------------------- building blocks
@pytest.mark.parametrize("n,b_mn_major,a_tmem", [(64, 0, 0), (128, 0, 0), (128, 1, 0),
                                                 (64, 0, 1), (128, 0, 1), (128, 1, 1)])
def test_fp8_mma_one_tile(n, b_mn_major, a_tmem):
    """E4M3 tcgen05 products (K-major / MN-major B, A from shared or tensor memory)
    against a CPU matmul of the decoded values."""
    g = torch.Generator().manual_seed(31 * n + 7 * b_mn_major + a_tmem)
    a = (torch.randn(128, 128, generator=g) * 8).to(torch.float8_e4m3fn)
    b = (torch.randn(n, 128, generator=g) * 8).to(torch.float8_e4m3fn)   # N x K
    b_dev = (u8(b).t().contiguous() if b_mn_major else u8(b)).cuda()
    a_dev = a.to(torch.float32).cuda() if a_tmem else u8(a).cuda()
    c = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    _capi.check(_capi.fa_selftest_umma_f8(a_dev, b_dev, c, n, b_mn_major, a_tmem), "umma_f8")
    torch.cuda.synchronize()
    ad, bd = a.to(torch.float64), b.to(torch.float64)
    ref = ad @ bd.t()
    scale = (ad.abs() @ bd.abs().t()).max().item()
    err = (c.cpu().double() - ref).abs().max().item()
    assert err <= 1e-6 * scale, (err, scale)


def test_fp8_pack_rounds_to_nearest_even_in_byte_order():
    """Off-grid fp32 A packed on the device (four per TMEM column) equals torch's
    E4M3 rounding of A, in the right byte order."""
    g = torch.Generator().manual_seed(5)
    a = torch.randn(128, 128, generator=g) * 20
    a[:, 0::4] *= 0.01                       # bytes of different size in each word
    b = (torch.randn(128, 128, generator=g) * 4).to(torch.float8_e4m3fn)
    c = torch.full((128, 128), float("nan"), dtype=torch.float32, device="cuda")
    _capi.check(_capi.fa_selftest_umma_f8(a.cuda(), u8(b).cuda(), c, 128, 0, 1), "umma_f8")
    torch.cuda.synchronize()
    ad = a.to(torch.float8_e4m3fn).to(torch.float64)
    bd = b.to(torch.float64)
    ref = ad @ bd.t()
    scale = (ad.abs() @ bd.abs().t()).max().item()
    assert (c.cpu().double() - ref).abs().max().item() <= 1e-6 * scale


# ---------------------------------------------------------------- the forward
def run_fp8(q8, k8, v8, causal, scale, ds):
    B, H, Sq, d = q8.shape
    Sk = k8.shape[2]
    qd, kd, vd = u8(q8).cuda(), u8(k8).cuda(), u8(v8).cuda()
    o_buf, l_buf = alloc_outputs(B, H, Sq, d)
    o, lse = views(o_buf, l_buf, B, H, Sq, d)
    stream = torch.cuda.current_stream()
    _capi.check(_capi.fa_forward_fp8(qd, kd, vd, o, lse, B, H, Sq, Sk, d, causal, scale, ds[0],
                                     ds[1], ds[2], stream), "fa_forward_fp8")
    torch.cuda.synchronize()
    _capi.check(_capi.fa_device_status(stream), "device status")
    check_guard(o_buf, l_buf, B, H, Sq, d)
    return o.float().cpu(), lse.cpu()


FP8_CASES = [
    # B, H, Sq, Sk, causal, q_factor
    (1, 1, 256, 256, False, 1.0),
    (1, 1, 256, 256, True, 1.0),
    (1, 2, 300, 300, True, 1.0),      # ragged tail
    (2, 2, 200, 520, True, 1.0),      # Sq < Sk: bottom-right offset
    (1, 2, 520, 200, True, 1.0),      # Sk < Sq: rows with no visible key
    (1, 1, 1, 300, False, 1.0),       # a single query row
    (1, 3, 700, 1100, False, 1.0),
    (2, 4, 1024, 1024, True, 4.0),    # large logits: the reference moves often
]


@pytest.mark.parametrize("case", FP8_CASES,
                         ids=lambda c: "b{}h{}q{}k{}{}x{:g}".format(*c[:4], "c" if c[4] else "n", c[5]))
def test_fp8_forward_parity(case):
    B, H, Sq, Sk, causal, qf = case
    w = custom(B, H, Sq, Sk, 128, causal, seed=B * 1000 + Sq + Sk, q_factor=qf)
    q8, k8, v8, ds = make_qkv_fp8(w)
    o, lse = run_fp8(q8, k8, v8, causal, w.scale, ds)
    o_ref, lse_ref = oracle.attention_fp8(q8, k8, v8, causal, w.scale, ds)
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("mult", [(0.5, 2.0, 4.0), (3.0, 0.125, 0.75)])
def test_fp8_descales(mult):
    """q and k descales scale the scores, v's scales O (non-power-of-two included).
    The O bar is absolute for unit-scale V, so O is compared divided by V's
    multiplier (bf16 rounding of O grows with |O|)."""
    w = custom(1, 2, 384, 384, 128, True, seed=77)
    q8, k8, v8, ds = make_qkv_fp8(w)
    ds = tuple(a * m for a, m in zip(ds, mult))
    o, lse = run_fp8(q8, k8, v8, True, w.scale, ds)
    o_ref, lse_ref = oracle.attention_fp8(q8, k8, v8, True, w.scale, ds)
    compare(o / mult[2], lse, o_ref / mult[2], lse_ref)


def test_fp8_within_rounding_bound_of_the_definition():
    """Against the unrounded definition: |o - o_def| <= 2^-4 sum_j P_j |v_j| (E4M3
    rounding of the weights) + 2e-2 (the bf16 bar for the rest), row by row."""
    w = custom(1, 1, 256, 256, 128, True, seed=3)
    q8, k8, v8, ds = make_qkv_fp8(w)
    o, _ = run_fp8(q8, k8, v8, True, w.scale, ds)
    o_def, _ = oracle.attention_fp8(q8, k8, v8, True, w.scale, ds, quantize_p=False)
    qb = (q8.to(torch.float32) * ds[0]).to(torch.bfloat16)
    kb = (k8.to(torch.float32) * ds[1]).to(torch.bfloat16)
    vabs = (v8.to(torch.float64) * ds[2]).abs().numpy()[0, 0]
    for i in range(w.Sq):
        P = oracle.probs_row(qb, kb, True, w.scale, 0, 0, i)
        bound = 2.0 ** -4 * (P @ vabs) + 2e-2
        assert np.all(np.abs(o[0, 0, i].numpy() - o_def[0, 0, i]) <= bound), i


def test_fp8_is_deterministic():
    w = custom(1, 4, 640, 640, 128, True, seed=8)
    q8, k8, v8, ds = make_qkv_fp8(w)
    o1, l1 = run_fp8(q8, k8, v8, True, w.scale, ds)
    o2, l2 = run_fp8(q8, k8, v8, True, w.scale, ds)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_rejects_bad_arguments():
    B, H, S = 1, 1, 128
    q = torch.zeros((B, H, S, 128), dtype=torch.uint8, device="cuda")
    o = torch.empty((B, H, S, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    f = _capi.fa_forward_fp8
    assert f(q, q, q, o, lse, B, H, S, S, 64, True, 0.1, 1, 1, 1) == _capi.FA_ERR_UNSUPPORTED
    assert f(q, q, q, o, lse, B, H, S, S, 128, True, 0.1, 0.0, 1, 1) == _capi.FA_ERR_UNSUPPORTED
    assert f(q, q, q, o, lse, B, H, S, S, 128, True, 0.1, 1, -1, 1) == _capi.FA_ERR_UNSUPPORTED
    assert f(q, q, q, o, lse, B, H, S, S, 128, True, 0.1, 1, 1, float("nan")) == \
        _capi.FA_ERR_INVALID_ARG
    assert f(q, q, q, o, lse, B, H, S, S, 128, True, float("inf"), 1, 1, 1) == \
        _capi.FA_ERR_INVALID_ARG
    assert f(q.view(-1)[1:], q, q, o, lse, B, H, S - 1, S, 128, True, 0.1, 1, 1, 1) == \
        _capi.FA_ERR_UNSUPPORTED                          # q not 16-byte aligned
    assert f(None, q, q, o, lse, B, H, S, S, 128, True, 0.1, 1, 1, 1) == _capi.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_fp8_headline_shape_sampled_rows():
    """B4 H32 S8192 d128 causal in E4M3, the launch the benchmark times, on sampled rows."""
    w = WORKLOADS[HEADLINE]
    q8, k8, v8, ds = make_qkv_fp8(w)
    o, lse = run_fp8(q8, k8, v8, True, w.scale, ds)
    rows = sample_rows(w, n_total=96)
    o_ref, lse_ref = oracle.attention_fp8(q8, k8, v8, True, w.scale, ds, rows=rows)
    og, lg = gather_rows(o, lse, rows)
    compare(og, lg, o_ref, lse_ref)
