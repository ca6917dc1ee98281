"""Pins for the FP8 forward of the oracle (E4M3 inputs, P rounded to E4M3).

Each pin checks the oracle against something other than itself:
  * the E4M3 decode and rounding against torch's float8_e4m3fn casts (a
    library routine) on every code and on values at and between grid points,
    plus closed forms of the format (largest finite 448, subnormal step 2^-9);
  * the unrounded FP8 forward against the bf16 oracle (already pinned) on the
    same decoded values, which torch decodes;
  * the rounded forward against the rounding bound that follows from E4M3's
    three mantissa bits;
  * a closed form for identical keys, where the rounded weights make the
    output (P_hat / p) * mean(v);
  * a hand-worked two-key example whose weights sit on the E4M3 grid.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_03_gb300.inputs import custom, make_qkv_fp8

LN2 = math.log(2.0)


def torch_decode(codes):
    t = torch.as_tensor(np.asarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_round(y32):
    return torch.as_tensor(np.asarray(y32, dtype=np.float32)).to(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.e4m3_decode(codes), torch_decode(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.isnan(ours).sum() == 2  # S.1111.111 only


def test_decode_closed_forms():
    """Bias 7, three mantissa bits, subnormals m/8 * 2^-6, no infinities."""
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0xB8: -1.0,
             0xFE: -448.0, 0x80: -0.0}
    got = oracle.e4m3_decode(list(cases))
    assert got.tolist() == list(cases.values())


def _grid():
    pos = torch_decode(np.arange(0x00, 0x7F, dtype=np.uint8))  # 0 .. 448, increasing
    assert np.all(np.diff(pos) > 0)
    return pos


def test_round_matches_torch_at_and_between_grid_points():
    pos = _grid()
    mids = 0.5 * (pos[1:] + pos[:-1])          # exact ties: fp32 holds them
    g = np.random.default_rng(7)
    mags = np.exp2(g.uniform(-12, math.log2(448.0), 20000))
    ys = np.concatenate([pos, mids, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20), mags])
    ys = np.concatenate([ys, -ys]).astype(np.float32)
    ours = oracle.e4m3_round(ys.astype(np.float64))
    ref = torch_round(ys)
    assert np.array_equal(ours, ref)


def test_round_error_bound_and_clamp():
    g = np.random.default_rng(8)
    y = np.exp2(g.uniform(-6, math.log2(448.0), 50000))
    r = oracle.e4m3_round(y)
    assert np.all(np.abs(r - y) <= 2.0 ** -4 * y)
    ys = np.exp2(g.uniform(-14, -6, 5000))
    assert np.all(np.abs(oracle.e4m3_round(ys) - ys) <= 2.0 ** -10)
    assert oracle.e4m3_round([1000.0, -600.0, 449.0]).tolist() == [448.0, -448.0, 448.0]
    grid = _grid()
    assert np.array_equal(oracle.e4m3_round(grid), grid)  # idempotent on the grid


SHAPES = [
    # B, H, Sq, Sk, d, causal
    (1, 1, 9, 9, 16, True),
    (1, 2, 5, 13, 32, True),      # bottom-right offset
    (2, 1, 9, 4, 16, True),       # Sk < Sq: rows with no visible key
    (1, 1, 7, 21, 64, False),
]


def fp8_case(B, H, Sq, Sk, d, causal, seed=0, factor=1.0):
    w = custom(B, H, Sq, Sk, d, causal, seed=seed, q_factor=factor)
    q8, k8, v8, ds = make_qkv_fp8(w)
    return w, q8, k8, v8, ds


def decoded_bf16(t8, ds):
    """torch's decode times the descale; exact in bf16 (3-bit mantissas, power-of-two descale)."""
    x = t8.to(torch.float32) * ds
    xb = x.to(torch.bfloat16)
    assert torch.equal(xb.to(torch.float32), x)
    return xb


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("descale", [None, (0.25, 2.0, 0.5)])
def test_unrounded_fp8_equals_bf16_definition(shape, descale):
    w, q8, k8, v8, ds = fp8_case(*shape, seed=5, factor=2.0)
    if descale is not None:
        ds = tuple(a * b for a, b in zip(ds, descale))
    o8, l8 = oracle.attention_fp8(q8, k8, v8, w.causal, w.scale, ds, quantize_p=False)
    ob, lb = oracle.attention(decoded_bf16(q8, ds[0]), decoded_bf16(k8, ds[1]),
                              decoded_bf16(v8, ds[2]), w.causal, w.scale)
    np.testing.assert_allclose(o8, ob, rtol=0, atol=1e-12)
    fin = np.isfinite(lb)
    assert np.array_equal(np.isfinite(l8), fin)
    np.testing.assert_allclose(l8[fin], lb[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
def test_rounded_weights_stay_within_the_e4m3_bound(shape):
    """|P_hat_j - p_j| <= 2^-4 p_j + 2^-17 (relative to a max weight in (1/2, 1]), so
    |o_hat - o| <= 2^-4 sum_j P_j |v_j| + 2^-16 sum_j |v_j| with P the softmax row."""
    w, q8, k8, v8, ds = fp8_case(*shape, seed=6, factor=3.0)
    oq, lq = oracle.attention_fp8(q8, k8, v8, w.causal, w.scale, ds, quantize_p=True)
    od, ld = oracle.attention_fp8(q8, k8, v8, w.causal, w.scale, ds, quantize_p=False)
    qb, kb, vb = decoded_bf16(q8, ds[0]), decoded_bf16(k8, ds[1]), decoded_bf16(v8, ds[2])
    vabs = vb.to(torch.float64).abs().numpy()
    worst = 0.0
    for b in range(w.B):
        for h in range(w.H):
            for i in range(w.Sq):
                P = oracle.probs_row(qb, kb, w.causal, w.scale, b, h, i)
                bound = 2.0 ** -4 * (P @ vabs[b, h]) + 2.0 ** -16 * vabs[b, h][P > 0].sum(0)
                err = np.abs(oq[b, h, i] - od[b, h, i])
                assert np.all(err <= bound + 1e-12), (b, h, i)
                worst = max(worst, float(err.max()))
    assert worst > 1e-6  # the rounding did happen
    fin = np.isfinite(ld)
    np.testing.assert_allclose(lq[fin], ld[fin], rtol=0, atol=1e-12)  # l is taken before rounding


@pytest.mark.parametrize("kcode", [0x30, 0x3B, 0x44, 0xB5])
def test_identical_keys_closed_form(kcode):
    """All keys equal: every x_j = x, so the rounded weights are all P_hat = 2^-7 e4m3(2^7 2^(x-M))
    against l = n 2^(x-M): the output is (P_hat / 2^(x-M)) * mean(v) over the visible keys."""
    Sq, Sk, d = 3, 10, 16
    g = torch.Generator().manual_seed(11)
    q8 = (torch.randn((1, 1, Sq, d), generator=g) * 4).to(torch.float8_e4m3fn)
    kb = torch.full((1, 1, Sk, d), kcode, dtype=torch.uint8)
    k8 = kb.view(torch.float8_e4m3fn)
    v8 = (torch.randn((1, 1, Sk, d), generator=g) * 8).to(torch.float8_e4m3fn)
    scale = 0.3
    o, lse = oracle.attention_fp8(q8, k8, v8, True, scale, (1.0, 1.0, 1.0), quantize_p=True)
    qd = q8.to(torch.float64)[0, 0]
    kd = k8.to(torch.float64)[0, 0, 0]
    vd = v8.to(torch.float64)[0, 0]
    for i in range(Sq):
        n = i + Sk - Sq + 1
        s = float(torch.tensor(scale, dtype=torch.float32)) * float(qd[i] @ kd)
        x = s / LN2
        p = 2.0 ** (x - math.ceil(x))
        p_hat = float(torch_round([2.0 ** 7 * p])[0]) / 2.0 ** 7
        expect = (p_hat / p) * vd[:n].mean(0).numpy()
        np.testing.assert_allclose(o[0, 0, i], expect, rtol=1e-12, atol=1e-12)
        assert abs(lse[0, 0, i] - (s + math.log(n))) < 1e-12


def test_two_key_hand_example():
    """q = 1, keys 1 and 0.5, values 2 and 4, scale 1, d = 1 (all exact in E4M3).
    x = (1, 0.5) / ln 2 = (1.4427, 0.7213); M = 2; 2^7 2^(x - M) = (86.98, 52.76).
    On the E4M3 grid 86.98 lies in [64, 128) with step 8 -> 88, and 52.76 in [32, 64)
    with step 4 -> 52, so P_hat = (88, 52) / 128 while l = 2^(x0-2) + 2^(x1-2)."""
    q8 = torch.tensor([0x38], dtype=torch.uint8).view(torch.float8_e4m3fn).reshape(1, 1, 1, 1)
    k8 = torch.tensor([0x38, 0x30], dtype=torch.uint8).view(torch.float8_e4m3fn).reshape(1, 1, 2, 1)
    v8 = torch.tensor([0x40, 0x48], dtype=torch.uint8).view(torch.float8_e4m3fn).reshape(1, 1, 2, 1)
    assert v8.to(torch.float32).flatten().tolist() == [2.0, 4.0]
    o, lse = oracle.attention_fp8(q8, k8, v8, False, 1.0, (1.0, 1.0, 1.0), quantize_p=True)
    l = 2.0 ** (1 / LN2 - 2) + 2.0 ** (0.5 / LN2 - 2)
    assert abs(o[0, 0, 0, 0] - (88 / 128 * 2 + 52 / 128 * 4) / l) < 1e-12
    assert abs(o[0, 0, 0, 0] - 2.74788) < 1e-5  # 3 / 1.09175, by hand
    assert abs(lse[0, 0, 0] - math.log(math.e + math.exp(0.5))) < 1e-12
    o0, _ = oracle.attention_fp8(q8, k8, v8, False, 1.0, (1.0, 1.0, 1.0), quantize_p=False)
    w0 = math.e / (math.e + math.exp(0.5))
    assert abs(o0[0, 0, 0, 0] - (2 * w0 + 4 * (1 - w0))) < 1e-12


def test_rows_entry_point_matches_full():
    w, q8, k8, v8, ds = fp8_case(2, 2, 11, 17, 32, True, seed=9)
    o, lse = oracle.attention_fp8(q8, k8, v8, True, w.scale, ds)
    rows = [(1, 0, 10), (0, 1, 0), (1, 1, 5), (0, 0, 7)]
    orr, lr = oracle.attention_fp8(q8, k8, v8, True, w.scale, ds, rows=rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(orr[n], o[b, h, i])
        assert lr[n] == lse[b, h, i]
