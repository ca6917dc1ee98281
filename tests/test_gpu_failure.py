"""Failure detection on the production kernels, without faulting or hanging a GPU.

fa_testing_stall_next_launch makes the next launch of the prefill kernel (or of
the split-KV verify kernel) skip one ring load in its first CTA, with a short
limit on every bounded wait of that launch. The consumer's wait for the missing
load then runs out, and the kernel's abort path runs for real: the CTA raises
its abort flag and records FA_ERR_TIMEOUT in the device status word, stops
issuing, drains the copies and MMAs it has in flight, frees its tensor memory
and returns; the other CTAs finish or give up at their next slow wait. Each
test checks that the host reads the timeout, that the call returned within a
few wait limits (no wait fell back to the 2 s default), and that the launches
after it on the same stream are correct: the next one, and the one 1024
launches later that takes the stalled launch's work-counter slot again (the
prefill kernel's counters are used in turn), which shows the counter went back
to zero. Tensor memory left allocated by the aborted CTA would have stalled
every later launch on its SM at its allocation.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import custom, make_qkv, sample_rows
from parity import compare, gather_rows

pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000_000  # 50 ms per bounded wait in the stalled launch


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _capi.load()


def _stalled(launch, kernel, skip):
    """Run `launch` once with a stall requested; returns (status, seconds)."""
    assert _capi.fa_device_status() == _capi.FA_OK
    _capi.check(_capi.fa_testing_stall_next_launch(kernel, skip, LIMIT_NS), "stall request")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _capi.check(launch(), "stalled launch")
    st = _capi.fa_device_status()  # synchronises the stream, reads and clears the word
    dt = time.perf_counter() - t0
    return st, dt


def test_the_stall_request_is_validated():
    f = _capi.fa_testing_stall_next_launch
    assert f(3, 0, LIMIT_NS) == _capi.FA_ERR_INVALID_ARG
    assert f(_capi.STALL_PREFILL, -1, LIMIT_NS) == _capi.FA_ERR_INVALID_ARG
    assert f(_capi.STALL_PREFILL, 0, 10) == _capi.FA_ERR_INVALID_ARG
    assert f(_capi.STALL_VERIFY, 0, 20_000_000_000) == _capi.FA_ERR_INVALID_ARG


def test_stalled_prefill_launch_reports_a_timeout_and_later_launches_are_correct():
    # 512 items for at most 152 CTAs: the first CTA has work, and its first
    # item loads K_0 then V_0 (ring load 1, the one skipped).
    w = custom(1, 64, 2048, 2048, 128, True, seed=23)
    q, k, v = make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device="cuda")

    def launch():
        return _capi.fa_prefill_forward(qd, kd, vd, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, True,
                                        w.scale)

    _capi.check(launch(), "first launch")
    torch.cuda.synchronize()
    o0, l0 = o.clone(), lse.clone()
    o.fill_(float("nan"))

    st, dt = _stalled(launch, _capi.STALL_PREFILL, 1)
    assert st == _capi.FA_ERR_TIMEOUT
    assert LIMIT_NS * 1e-9 <= dt < 1.5, dt
    assert _capi.fa_device_status() == _capi.FA_OK   # read and cleared

    _capi.check(launch(), "launch after the stall")
    torch.cuda.synchronize()
    assert _capi.fa_device_status() == _capi.FA_OK
    assert torch.equal(o, o0) and torch.equal(lse, l0)

    for _ in range(1024):  # the last of these takes the stalled launch's counter slot
        o.fill_(float("nan"))
        _capi.check(launch(), "launch")
    torch.cuda.synchronize()
    assert _capi.fa_device_status() == _capi.FA_OK
    assert torch.equal(o, o0) and torch.equal(lse, l0)
    rows = sample_rows(w, n_total=48)
    ro, rl = oracle.attention(q, k, v, True, w.scale, rows=rows)
    og, lg = gather_rows(o.float().cpu(), lse.cpu(), rows)
    compare(og, lg, ro, rl)


@pytest.mark.parametrize("n_split", [1, 3])
def test_stalled_verify_launch_reports_a_timeout_and_the_next_launch_is_correct(n_split):
    w = custom(2, 4, 5, 1000, 128, True, seed=29)
    q, k, v = make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device="cuda")
    need = _capi.fa_verify_workspace_size(w.B, w.H, w.Sq, w.Sk, w.d, n_split)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")

    def launch():
        return _capi.fa_verify_forward(qd, kd, vd, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, True,
                                       w.scale, n_split, ws, need)

    st, dt = _stalled(launch, _capi.STALL_VERIFY, 2)
    assert st == _capi.FA_ERR_TIMEOUT
    assert LIMIT_NS * 1e-9 <= dt < 1.5, dt
    assert _capi.fa_device_status() == _capi.FA_OK

    o.fill_(float("nan"))
    _capi.check(launch(), "launch after the stall")
    torch.cuda.synchronize()
    assert _capi.fa_device_status() == _capi.FA_OK
    ro, rl = oracle.attention(q, k, v, True, w.scale)
    compare(o.float().cpu(), lse.cpu(), ro, rl)
