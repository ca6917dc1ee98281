"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it, element by element, with the fp64 oracle on the same bf16 inputs.

Tolerances (bf16 inputs and output, fp32 accumulation, against fp64):
O max-abs <= 2e-2, O mean-abs <= 2e-3, LSE abs <= 1e-3; fully masked rows must
be exactly O = 0 and LSE = -inf on both sides.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_tiled_attention_03_gb300 import _capi

TOL_O_MAX = 2e-2
TOL_O_MEAN = 2e-3
TOL_LSE = 1e-3

GUARD = 64  # poisoned elements after each output buffer


def alloc_outputs(B, H, Sq, d, device="cuda"):
    """O and LSE with a poisoned guard band after them (checked by check_guard)."""
    o_buf = torch.full((B * H * Sq * d + GUARD,), float("nan"), dtype=torch.bfloat16, device=device)
    l_buf = torch.full((B * H * Sq + GUARD,), 12345.0, dtype=torch.float32, device=device)
    o_buf[: B * H * Sq * d].fill_(float("nan"))
    return o_buf, l_buf


def views(o_buf, l_buf, B, H, Sq, d):
    return o_buf[: B * H * Sq * d].view(B, H, Sq, d), l_buf[: B * H * Sq].view(B, H, Sq)


def check_guard(o_buf, l_buf, B, H, Sq, d):
    tail_o = o_buf[B * H * Sq * d:]
    tail_l = l_buf[B * H * Sq:]
    assert torch.isnan(tail_o.float()).all(), "kernel wrote past the end of O"
    assert (tail_l == 12345.0).all(), "kernel wrote past the end of LSE"


def run(entry: str, q, k, v, causal: bool, scale: float, n_split: int | None = None,
        workspace=None):
    """Run one C entry point on CUDA copies of q, k, v. Returns (o, lse) on the CPU."""
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_buf, l_buf = alloc_outputs(B, H, Sq, d)
    o, lse = views(o_buf, l_buf, B, H, Sq, d)
    stream = torch.cuda.current_stream()
    if entry == "fa_forward":
        st = _capi.fa_forward(qd, kd, vd, o, lse, B, H, Sq, Sk, d, causal, scale, stream)
    elif entry == "fa_prefill_forward":
        st = _capi.fa_prefill_forward(qd, kd, vd, o, lse, B, H, Sq, Sk, d, causal, scale, stream)
    elif entry == "fa_reference_forward_simt":
        st = _capi.fa_reference_forward_simt(qd, kd, vd, o, lse, B, H, Sq, Sk, d, causal, scale,
                                             stream)
    elif entry == "fa_verify_forward":
        ns = n_split or 0
        need = _capi.fa_verify_workspace_size(B, H, Sq, Sk, d, ns)
        ws = workspace
        if ws is None and need:
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        st = _capi.fa_verify_forward(qd, kd, vd, o, lse, B, H, Sq, Sk, d, causal, scale, ns, ws,
                                     need if ws is not None else 0, stream)
    elif entry == "fa_forward_ws":
        need = _capi.fa_workspace_size(B, H, Sq, Sk, d)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        st = _capi.fa_forward_ws(qd, kd, vd, o, lse, B, H, Sq, Sk, d, causal, scale, ws, need,
                                 stream)
    else:
        raise ValueError(entry)
    _capi.check(st, entry)
    torch.cuda.synchronize()
    _capi.check(_capi.fa_device_status(stream), "device status")
    check_guard(o_buf, l_buf, B, H, Sq, d)
    return o.float().cpu(), lse.cpu()


def compare(o_gpu, lse_gpu, o_ref, lse_ref):
    """Element-wise comparison; returns the error summary (asserts the bar)."""
    og = np.asarray(o_gpu, dtype=np.float64)
    lg = np.asarray(lse_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64).reshape(og.shape)
    lse_ref = np.asarray(lse_ref, dtype=np.float64).reshape(lg.shape)
    assert np.all(np.isfinite(og)), "non-finite O"
    masked = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), masked), "fully masked rows differ"
    err = np.abs(og - o_ref)
    lerr = np.abs(lg[~masked] - lse_ref[~masked]) if (~masked).any() else np.zeros(1)
    summary = dict(o_max=float(err.max()), o_mean=float(err.mean()), lse_max=float(lerr.max()))
    if masked.any():
        assert np.all(og[masked] == 0.0), "fully masked rows must give O = 0"
    assert summary["o_max"] <= TOL_O_MAX, summary
    assert summary["o_mean"] <= TOL_O_MEAN, summary
    assert summary["lse_max"] <= TOL_LSE, summary
    return summary


def oracle_full(q, k, v, causal, scale):
    return oracle.attention(q, k, v, causal, scale)


def oracle_rows(q, k, v, causal, scale, rows):
    return oracle.attention(q, k, v, causal, scale, rows=rows)


def gather_rows(o, lse, rows):
    idx = torch.tensor(rows, dtype=torch.long)
    return (o[idx[:, 0], idx[:, 1], idx[:, 2]].numpy(), lse[idx[:, 0], idx[:, 1], idx[:, 2]].numpy())
