"""The debug build (FA_DEBUG): device-side index checks on the kernels' paged,
persistent and split paths, standing in for a memory checker.

The debug library is the same sources compiled with FA_DEBUG: before each
plain global load or store a kernel checks the index it computed (and skips the
access if the check fails), and it checks the start coordinates of its TMA
copies (reported only). A failed check sets a bit in the device status word,
which fa_device_status reports as FA_ERR_BOUNDS; nothing asserts or traps.

The tests check that a failing check is reported (and that the release build
compiles checks away), then run every kernel of the debug library on edge shapes
(ragged tiles, Sq < Sk and Sk < Sq, d = 64 and 128, several split counts,
draft-tree masks, paged caches with short sequences and unread garbage table
entries, the backward, FP8) and require no failed check and outputs identical,
bit for bit, to the release library's.
"""
import contextlib

import pytest
import torch

from exact_tiled_attention_03_gb300 import _capi, build
from exact_tiled_attention_03_gb300.inputs import (custom, make_paged_kv, make_qkv, make_qkv_fp8,
                                                   make_tree_masks)
from test_gpu_backward import run_fwd_bwd, upstream
from test_gpu_fp8 import run_fp8
from test_gpu_verify_ext import run_paged, run_verify_tree
from parity import run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    release = _capi.load()
    debug = _capi.open_library(build.build_debug())
    return release, debug


@contextlib.contextmanager
def using(lib):
    saved = _capi._lib
    _capi._lib = lib
    try:
        yield
    finally:
        _capi._lib = saved


def both(libs, fn):
    """fn() through the release library, then through the debug library, whose
    checks must all pass; the outputs must be identical."""
    release, debug = libs
    with using(release):
        a = fn()
        assert _capi.fa_device_status() == _capi.FA_OK
    with using(debug):
        assert _capi.fa_device_status() == _capi.FA_OK
        b = fn()
        torch.cuda.synchronize()
        assert _capi.fa_device_status() == _capi.FA_OK, "an index check failed"
    for x, y in zip(a, b):
        x, y = torch.as_tensor(x), torch.as_tensor(y)
        assert torch.equal(x, y) or (x.is_floating_point() and torch.equal(torch.nan_to_num(x),
                                                                           torch.nan_to_num(y)))


def test_a_failed_check_is_reported_and_release_builds_have_none(libs):
    release, debug = libs
    assert debug.fa_testing_debug_checks() == 1 and release.fa_testing_debug_checks() == 0
    with using(debug):
        assert _capi.fa_device_status() == _capi.FA_OK
        _capi.check(_capi.fa_selftest_index_check(0), "passing check")
        assert _capi.fa_device_status() == _capi.FA_OK
        _capi.check(_capi.fa_selftest_index_check(1), "failing check")
        assert _capi.fa_device_status() == _capi.FA_ERR_BOUNDS
        assert _capi.fa_device_status() == _capi.FA_OK   # read and cleared
    with using(release):
        _capi.check(_capi.fa_selftest_index_check(1), "failing check, compiled away")
        assert _capi.fa_device_status() == _capi.FA_OK


@pytest.mark.parametrize("case", [(1, 2, 300, 300, 128, True), (1, 1, 200, 520, 128, True),
                                  (1, 2, 300, 100, 64, True), (2, 1, 257, 700, 64, False),
                                  (1, 1, 1, 1, 128, False)],
                         ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
def test_prefill_debug_build(libs, case):
    B, H, Sq, Sk, d, causal = case
    w = custom(B, H, Sq, Sk, d, causal, seed=Sq + Sk, q_factor=2.0)
    q, k, v = make_qkv(w)
    both(libs, lambda: run("fa_prefill_forward", q, k, v, causal, w.scale))


@pytest.mark.parametrize("case", [(2, 4, 5, 1000, 128, 1), (2, 4, 5, 1000, 128, 3),
                                  (1, 3, 16, 700, 64, 0), (3, 2, 1, 64, 128, 1)],
                         ids=lambda c: "b{}h{}q{}k{}d{}s{}".format(*c))
def test_verify_debug_build(libs, case):
    B, H, Sq, Sk, d, ns = case
    w = custom(B, H, Sq, Sk, d, True, seed=Sq * 3 + Sk)
    q, k, v = make_qkv(w)
    both(libs, lambda: run("fa_verify_forward", q, k, v, True, w.scale, n_split=ns))


def test_verify_tree_debug_build(libs):
    B, H, Sq, Sk, d = 2, 3, 5, 300, 128
    w = custom(B, H, Sq, Sk, d, True, seed=41)
    q, k, v = make_qkv(w)
    masks = make_tree_masks(B, Sq, seed=Sk)
    both(libs, lambda: run_verify_tree(q, k, v, masks, w.scale, 3))


@pytest.mark.parametrize("page_size", [16, 32, 64])
def test_verify_paged_debug_build(libs, page_size):
    B, H, Sq, d, Smax = 4, 3, 5, 128, 700
    lens = [700, 5, 333, 64]
    w = custom(B, H, Sq, Smax, d, True, seed=page_size)
    q, k, v = make_qkv(w)
    kp, vp, table, lens_t = make_paged_kv(k, v, lens, page_size, seed=page_size)
    both(libs, lambda: run_paged(q, kp, vp, table, lens_t, page_size, Smax, True, None, w.scale, 5))


@pytest.mark.parametrize("case", [(1, 2, 300, 300, 128, True), (1, 1, 300, 100, 64, True),
                                  (1, 2, 200, 500, 128, False)],
                         ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
def test_backward_debug_build(libs, case):
    B, H, Sq, Sk, d, causal = case
    w = custom(B, H, Sq, Sk, d, causal, seed=Sq + 7 * Sk, q_factor=2.0)
    q, k, v = make_qkv(w)
    do = upstream(q, w.seed)
    both(libs, lambda: run_fwd_bwd(q, k, v, do, causal, w.scale))


@pytest.mark.parametrize("case", [(1, 2, 300, 300, True), (1, 2, 520, 200, True), (1, 1, 1, 300, False)],
                         ids=lambda c: "b{}h{}q{}k{}{}".format(*c[:4], "c" if c[4] else "n"))
def test_fp8_debug_build(libs, case):
    B, H, Sq, Sk, causal = case
    w = custom(B, H, Sq, Sk, 128, causal, seed=Sq * 5 + Sk)
    q8, k8, v8, ds = make_qkv_fp8(w)
    both(libs, lambda: run_fp8(q8, k8, v8, causal, w.scale, ds))
