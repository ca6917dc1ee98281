"""GPU parity at the largest sizes: tensors past 2^31 elements (every offset
the kernels form past that point must be 64-bit; the loads and stores go
through TMA coordinates) and the verify grid's (b, h) limit of 65535. Inputs
are drawn on the device (``make_qkv_device``); the oracle sees the sampled
heads, copied to the host, at the far end of each buffer."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import custom, make_qkv_device
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _capi.load()


def head(t, b, h):
    return t[b:b + 1, h:h + 1].cpu()


def forward(q, k, v, causal, scale):
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    _capi.check(_capi.fa_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale), "fa_forward")
    torch.cuda.synchronize()
    _capi.check(_capi.fa_device_status(), "device status")
    return o, lse


def test_prefill_past_2_31_elements():
    """B17 H128 S8192 d128 causal: 2.28e9 elements per tensor. Heads (16, 0) and
    (16, 127) start at and end past element 2^31."""
    w = custom(17, 128, 8192, 8192, 128, True, seed=51)
    assert w.B * w.H * w.Sq * w.d > 2 ** 31
    q, k, v = make_qkv_device(w)
    o, lse = forward(q, k, v, True, w.scale)
    rows = [0, 1, 127, 128, 4095, 4096, 8190, 8191]
    for b, h in ((0, 0), (16, 0), (16, 127)):
        ro, rl = oracle.attention(head(q, b, h), head(k, b, h), head(v, b, h), True, w.scale,
                                  rows=[(0, 0, i) for i in rows])
        compare(o[b, h, rows].float().cpu().numpy(), lse[b, h, rows].cpu().numpy(), ro, rl)


def test_backward_past_2_31_elements():
    """The backward at the same size: dQ, dK, dV rows of the last head."""
    w = custom(17, 128, 8192, 8192, 128, True, seed=52)
    q, k, v = make_qkv_device(w)
    g = torch.Generator(device="cuda").manual_seed(53)
    do = torch.empty_like(q)
    for b in range(w.B):
        do[b].copy_(torch.randn(q.shape[1:], generator=g, device="cuda"))
    o, lse = forward(q, k, v, True, w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B, H, S, d = q.shape
    _capi.check(_capi.fa_backward(q, k, v, o, lse, do, dq, dk, dv, B, H, S, S, d, True, w.scale,
                                  None, 0), "fa_backward")
    torch.cuda.synchronize()
    _capi.check(_capi.fa_device_status(), "device status")
    rows = [0, 127, 128, 4095, 8191]
    for b, h in ((16, 127),):
        rq, rk, rv = oracle.attention_backward_rows(head(q, b, h), head(k, b, h), head(v, b, h),
                                                    head(do, b, h), True, w.scale, 0, 0, rows, rows)
        for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            got = got[b, h, rows].float().cpu().numpy()
            assert np.all(np.isfinite(got)), name
            err = np.abs(got - ref)
            assert err.max() <= 2e-2 * np.max(np.abs(ref)) + 1e-4, (name, err.max())
            assert err.mean() <= 5e-3 * np.mean(np.abs(ref)) + 1e-5, (name, err.mean())


def test_verify_past_2_31_elements():
    """B32 H128 Sq5 Sk4352 d128 (split-KV path): 2.28e9 elements in K and in V."""
    w = custom(32, 128, 5, 4352, 128, True, seed=54)
    assert w.B * w.H * w.Sk * w.d > 2 ** 31
    q, k, v = make_qkv_device(w)
    o, lse = forward(q, k, v, True, w.scale)
    for b, h in ((0, 0), (31, 127), (20, 5)):
        ro, rl = oracle.attention(head(q, b, h), head(k, b, h), head(v, b, h), True, w.scale)
        compare(o[b:b + 1, h:h + 1].float().cpu().numpy(), lse[b:b + 1, h:h + 1].cpu().numpy(),
                ro, rl)


def test_verify_at_the_grid_limit_of_65535_heads():
    """B*H = 65535 runs (one CTA row per (b, h)); 65536 is rejected before any launch."""
    w = custom(65535, 1, 1, 64, 64, True, seed=55)
    q, k, v = make_qkv_device(w)
    o, lse = forward(q, k, v, True, w.scale)
    for b in (0, 40000, 65534):
        ro, rl = oracle.attention(head(q, b, 0), head(k, b, 0), head(v, b, 0), True, w.scale)
        compare(o[b:b + 1].float().cpu().numpy(), lse[b:b + 1].cpu().numpy(), ro, rl)
    del q, k, v, o, lse
    qs = torch.zeros((65536, 1, 1, 64), dtype=torch.bfloat16, device="cuda")
    ks = torch.zeros((65536, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    os_ = torch.empty_like(qs)
    ls = torch.empty((65536, 1, 1), device="cuda")
    assert _capi.fa_forward(qs, ks, ks, os_, ls, 65536, 1, 1, 64, 64, True, 0.125) == \
        _capi.FA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
