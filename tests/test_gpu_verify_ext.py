"""GPU parity of the split-KV verify path's extensions: draft-tree masks and a
paged KV cache read through a block table, against the fp64 oracle (masked
definition; per-sequence gathers of the logical K/V)."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import custom, make_paged_kv, make_qkv, make_tree_masks
from parity import compare

pytestmark = pytest.mark.gpu


def dense_visible(masks, Sq, Sk_list):
    """[B, Sq, max Sk] 0/1 visibility from the per-row draft masks (cache always visible)."""
    B = masks.shape[0]
    Smax = max(Sk_list)
    vis = np.zeros((B, Sq, Smax), np.uint8)
    for b in range(B):
        Sk = Sk_list[b]
        prefix = Sk - Sq
        for i in range(Sq):
            m = int(masks[b, i]) & 0xFFFFFFFF
            for j in range(Sk):
                vis[b, i, j] = 1 if j < prefix or (m >> (j - prefix)) & 1 else 0
    return vis


def run_verify_tree(q, k, v, masks, scale, n_split):
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    o = torch.full((B, H, Sq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Sq), float("nan"), device="cuda")
    need = _capi.fa_verify_workspace_size(B, H, Sq, Sk, d, n_split)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    _capi.check(_capi.fa_verify_tree_forward(q.cuda(), k.cuda(), v.cuda(), o, lse, B, H, Sq, Sk, d,
                                             masks.cuda(), scale, n_split, ws, need),
                "fa_verify_tree_forward")
    torch.cuda.synchronize()
    _capi.check(_capi.fa_device_status(), "device status")
    return o.float().cpu(), lse.cpu()


@pytest.mark.parametrize("case", [(2, 3, 5, 300, 128), (1, 2, 16, 1000, 64), (2, 2, 1, 130, 128),
                                  (1, 2, 8, 6, 128), (4, 2, 12, 4096, 128)],
                         ids=lambda c: "b{}h{}q{}k{}d{}".format(*c))
@pytest.mark.parametrize("n_split", [0, 1, 3])
def test_tree_mask_matches_masked_definition(case, n_split):
    B, H, Sq, Sk, d = case
    w = custom(B, H, Sq, Sk, d, True, seed=Sq * 13 + Sk, q_factor=2.0)
    q, k, v = make_qkv(w)
    masks = make_tree_masks(B, Sq, seed=Sk)
    if n_split > -(-Sk // 64):
        pytest.skip("more splits than 64-key chunks")
    o, lse = run_verify_tree(q, k, v, masks, w.scale, n_split)
    ro, rl = oracle.attention_masked(q, k, v, dense_visible(masks.numpy(), Sq, [Sk] * B), w.scale)
    compare(o, lse, ro, rl)


def test_chain_tree_equals_causal_verify():
    """The chain mask (bits 0..i) is the causal verify step, bit for bit."""
    w = custom(2, 4, 5, 1000, 128, True, seed=17)
    q, k, v = make_qkv(w)
    chain = torch.tensor([[(2 << i) - 1 for i in range(5)]] * 2, dtype=torch.int32)
    o_t, l_t = run_verify_tree(q, k, v, chain, w.scale, 4)
    o = torch.empty((2, 4, 5, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 4, 5), device="cuda")
    need = _capi.fa_verify_workspace_size(2, 4, 5, 1000, 128, 4)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    _capi.check(_capi.fa_verify_forward(q.cuda(), k.cuda(), v.cuda(), o, lse, 2, 4, 5, 1000, 128, 1,
                                        w.scale, 4, ws, need), "fa_verify_forward")
    torch.cuda.synchronize()
    assert torch.equal(o.float().cpu(), o_t) and torch.equal(lse.cpu(), l_t)


def run_paged(q, kp, vp, table, lens, page_size, max_len, causal, masks, scale, n_split):
    B, H, Sq, d = q.shape
    o = torch.full((B, H, Sq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Sq), float("nan"), device="cuda")
    need = _capi.fa_verify_workspace_size(B, H, Sq, max_len, d, n_split)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    _capi.check(_capi.fa_verify_paged_forward(
        q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(), o, lse, B, H, Sq, d,
        kp.shape[0], page_size, table.shape[1], max_len, causal,
        None if masks is None else masks.cuda(), scale, n_split, ws, need), "fa_verify_paged_forward")
    torch.cuda.synchronize()
    _capi.check(_capi.fa_device_status(), "device status")
    return o.float().cpu(), lse.cpu()


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("mode", ["causal", "tree", "noncausal"])
@pytest.mark.parametrize("n_split", [0, 1, 5])
def test_paged_kv_matches_per_sequence_oracle(page_size, mode, n_split):
    B, H, Sq, d, Smax = 4, 3, 5, 128, 700
    lens = [700, 5, 333, 64]                       # varied lengths, one equal to Sq
    w = custom(B, H, Sq, Smax, d, True, seed=page_size + n_split, q_factor=2.0)
    q, k, v = make_qkv(w)
    kp, vp, table, lens_t = make_paged_kv(k, v, lens, page_size, seed=page_size)
    masks = make_tree_masks(B, Sq, seed=7) if mode == "tree" else None
    o, lse = run_paged(q, kp, vp, table, lens_t, page_size, Smax, mode == "causal", masks,
                       w.scale, n_split)
    for b in range(B):
        Sk = lens[b]
        kb, vb, qb = k[b:b + 1, :, :Sk], v[b:b + 1, :, :Sk], q[b:b + 1]
        if mode == "tree":
            ro, rl = oracle.attention_masked(qb, kb, vb, dense_visible(masks[b:b + 1].numpy(), Sq, [Sk]),
                                             w.scale)
        else:
            ro, rl = oracle.attention(qb, kb, vb, mode == "causal", w.scale)
        compare(o[b:b + 1], lse[b:b + 1], ro, rl)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("n_split", [0, 3])
def test_paged_kv_head_dim_64(page_size, n_split):
    """d = 64 pages (128-byte rows: one box per page at every page size)."""
    B, H, Sq, d, Smax = 3, 2, 5, 64, 520
    lens = [520, 77, 200]
    w = custom(B, H, Sq, Smax, d, True, seed=31 * page_size + n_split)
    q, k, v = make_qkv(w)
    kp, vp, table, lens_t = make_paged_kv(k, v, lens, page_size, seed=page_size + 1)
    o, lse = run_paged(q, kp, vp, table, lens_t, page_size, Smax, True, None, w.scale, n_split)
    for b in range(B):
        Sk = lens[b]
        ro, rl = oracle.attention(q[b:b + 1], k[b:b + 1, :, :Sk], v[b:b + 1, :, :Sk], True, w.scale)
        compare(o[b:b + 1], lse[b:b + 1], ro, rl)


@pytest.mark.parametrize("page_size", [16, 32, 64])
def test_paged_kv_entries_outside_the_pool_read_as_zeros(page_size):
    """A block-table entry outside [0, num_pages) reads as zero K and V rows."""
    B, H, Sq, d, Smax = 2, 3, 5, 128, 700
    lens = [700, 333]
    w = custom(B, H, Sq, Smax, d, True, seed=41 + page_size)
    q, k, v = make_qkv(w)
    kp, vp, table, lens_t = make_paged_kv(k, v, lens, page_size, seed=page_size + 2)
    num_pages = kp.shape[0]
    table[0, 3] = num_pages + 3
    table[1, 1] = -1
    k_log, v_log = k.clone(), v.clone()
    for b, lp in ((0, 3), (1, 1)):
        k_log[b, :, lp * page_size:(lp + 1) * page_size] = 0
        v_log[b, :, lp * page_size:(lp + 1) * page_size] = 0
    o, lse = run_paged(q, kp, vp, table, lens_t, page_size, Smax, True, None, w.scale, 0)
    for b in range(B):
        Sk = lens[b]
        ro, rl = oracle.attention(q[b:b + 1], k_log[b:b + 1, :, :Sk], v_log[b:b + 1, :, :Sk], True,
                                  w.scale)
        compare(o[b:b + 1], lse[b:b + 1], ro, rl)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("d", [64, 128])
def test_paged_kv_with_contiguous_pages_equals_contiguous_path(page_size, d):
    """Pages laid out in order reproduce the contiguous verify kernel exactly,
    whatever box layout the page size selects."""
    B, H, S = 2, 4, 1024
    w = custom(B, H, 5, S, d, True, seed=29)
    q, k, v = make_qkv(w)
    P = page_size
    kp = k.reshape(B, H, S // P, P, d).permute(0, 2, 1, 3, 4).reshape(-1, H, P, d).contiguous()
    vp = v.reshape(B, H, S // P, P, d).permute(0, 2, 1, 3, 4).reshape(-1, H, P, d).contiguous()
    table = torch.arange(B * (S // P), dtype=torch.int32).reshape(B, S // P)
    lens = torch.tensor([S] * B, dtype=torch.int32)
    o_p, l_p = run_paged(q, kp, vp, table, lens, P, S, True, None, w.scale, 4)
    o = torch.empty((B, H, 5, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, 5), device="cuda")
    need = _capi.fa_verify_workspace_size(B, H, 5, S, d, 4)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    _capi.check(_capi.fa_verify_forward(q.cuda(), k.cuda(), v.cuda(), o, lse, B, H, 5, S, d, 1,
                                        w.scale, 4, ws, need), "fa_verify_forward")
    torch.cuda.synchronize()
    assert torch.equal(o.float().cpu(), o_p) and torch.equal(lse.cpu(), l_p)
