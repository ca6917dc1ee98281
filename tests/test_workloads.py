"""Host logic of the workload definitions: shape arithmetic, pair counts, seeds."""
import math

import pytest
import torch

from exact_tiled_attention_03_gb300.inputs import WORKLOADS, HEADLINE, VERIFY, custom, make_qkv, sample_rows
from golden_io import pages_numbers


@pytest.mark.parametrize("Sq,Sk,causal", [(1, 1, True), (7, 7, True), (5, 13, True), (13, 5, True),
                                          (3, 1, True), (1, 9, True), (6, 11, False), (128, 300, True)])
def test_visible_pairs_closed_form_matches_brute_force(Sq, Sk, causal):
    w = custom(1, 1, Sq, Sk, 8, causal)
    assert w.visible_pairs() == sum(w.visible_keys(i) for i in range(Sq))


def test_headline_flop_counts():
    w = WORKLOADS[HEADLINE]
    S = 8192
    assert w.visible_pairs() == S * (S + 1) // 2
    assert w.exact_flops() == 4 * 128 * (S * (S + 1) // 2) * 4 * 32
    assert abs(w.exact_flops() - 2.1993e12) / 2.1993e12 < 1e-4
    assert abs(w.fa_convention_flops() - 2.1990e12) / 2.1990e12 < 1e-4


def test_verify_shape_counts():
    w = WORKLOADS[VERIFY]
    # query i sees keys [0, 4091 + i]
    assert [w.visible_keys(i) for i in range(5)] == [4092, 4093, 4094, 4095, 4096]
    assert w.visible_pairs() == 20470
    assert abs(w.io_bytes() - 1.0751e9) / 1.0751e9 < 1e-3


def test_page_printed_sizes():
    """The score-matrix sizes the pages print, from the same shape arithmetic."""
    nums = pages_numbers()
    a = nums["score_matrix_8k"]["inputs"]
    w = custom(int(a["B"]), int(a["H"]), int(a["S"]), int(a["S"]), 128, True)
    assert round(w.score_matrix_bytes(int(a["elem_bytes"])) / 1e9, 1) == 17.2
    assert w.score_matrix_bytes() == WORKLOADS[HEADLINE].score_matrix_bytes()
    a = nums["score_matrix_32k"]["inputs"]
    w = custom(1, 1, int(a["S"]), int(a["S"]), 64, True)
    assert round(w.score_matrix_bytes(int(a["elem_bytes"])) / 1e9) == 2
    a = nums["decode_floor"]["inputs"]
    t = a["bytes"] / a["bandwidth"]
    assert round(t * 1e3, 1) == 4.8
    assert round(1 / t) == 209


def test_inputs_are_seeded_and_bf16():
    w = custom(1, 2, 9, 11, 16, True, seed=5)
    a = make_qkv(w)
    b = make_qkv(w)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.is_contiguous()
        assert torch.equal(x, y)
    assert a[0].shape == (1, 2, 9, 16) and a[1].shape == (1, 2, 11, 16)
    # stress variant: Q scaled by 4 before rounding
    ws = custom(1, 2, 9, 11, 16, True, seed=5, q_factor=4.0)
    qs = make_qkv(ws)[0]
    assert torch.equal(qs, make_qkv(ws)[0])
    assert qs.float().abs().max() > 2 * a[0].float().abs().max()


def test_device_inputs_are_seeded_and_bf16():
    """make_qkv_device (the generator of the largest GPU cases), run here with the
    CPU generator: seeded, bf16, contiguous, with the recipe's N(0, 1) statistics
    and q_factor."""
    from exact_tiled_attention_03_gb300 import inputs

    w = custom(3, 2, 64, 80, 16, True, seed=9)
    a = inputs.make_qkv_device(w, "cpu")
    b = inputs.make_qkv_device(w, "cpu")
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.is_contiguous() and torch.equal(x, y)
    assert a[0].shape == (3, 2, 64, 16) and a[1].shape == (3, 2, 80, 16)
    assert abs(float(a[1].float().std()) - 1.0) < 0.05 and abs(float(a[2].float().mean())) < 0.05
    q4 = inputs.make_qkv_device(custom(3, 2, 64, 80, 16, True, seed=9, q_factor=4.0), "cpu")[0]
    assert abs(float(q4.float().std()) / float(a[0].float().std()) - 4.0) < 0.1


def test_scale_is_fp32_of_inverse_sqrt_d():
    for d in (64, 128):
        w = custom(1, 1, 1, 1, d, False)
        assert w.scale == float(torch.tensor(1 / math.sqrt(d), dtype=torch.float32))


def test_sampled_rows_cover_tile_boundaries():
    w = WORKLOADS[HEADLINE]
    rows = sample_rows(w, n_total=64)
    assert len(rows) == 64
    ii = {i for _, _, i in rows}
    for i in (0, 127, 128, 8191):
        assert i in ii
    for b, h, i in rows:
        assert 0 <= b < w.B and 0 <= h < w.H and 0 <= i < w.Sq
    w2 = WORKLOADS["prefill_b1h32s32768d64_causal"]
    rows2 = sample_rows(w2, per_head=64)
    assert len(rows2) == 32 * 64
    assert {0, 32767, 127, 128, 255, 256} <= {i for _, _, i in rows2}
