"""The C ABI on a host without a GPU: the library loads, exports every entry
point the headers declare, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from exact_tiled_attention_03_gb300 import build, _capi
    build.build()
    return _capi


def declared_functions():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(fa_\w+)\s*\(", text, flags=re.M))
    return names


def test_headers_declare_the_expected_entry_points():
    names = declared_functions()
    for must in ("fa_forward", "fa_forward_ws", "fa_workspace_size", "fa_status_string",
                 "fa_device_status", "fa_prefill_forward", "fa_verify_forward"):
        assert must in names


def test_library_exports_every_declared_symbol(capi):
    lib = capi.load()
    out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(fa_\w+)$", out, flags=re.M))
    declared = declared_functions()
    assert declared <= exported, declared - exported
    assert set(capi.SIGNATURES) == declared
    for name in declared:
        assert getattr(lib, name) is not None


def test_status_strings(capi):
    for code in range(7):
        s = capi.fa_status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert capi.fa_status_string(0) == "ok"
    assert capi.fa_status_string(99) == "unknown status"


ALIGNED = 0x100000  # fake, 16-byte aligned addresses: validation never dereferences them


def call(capi, fn="fa_forward", q=ALIGNED, k=ALIGNED, v=ALIGNED, o=ALIGNED, lse=ALIGNED,
         B=1, H=1, Sq=256, Sk=256, d=128, causal=1, scale=0.125, **kw):
    f = getattr(capi, fn)
    if fn == "fa_verify_forward":
        return f(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, kw.get("n_split", 0),
                 kw.get("ws", None), kw.get("ws_bytes", 0), 0)
    if fn == "fa_forward_ws":
        return f(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, kw.get("ws", None),
                 kw.get("ws_bytes", 0), 0)
    return f(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, 0)


@pytest.mark.parametrize("fn", ["fa_forward", "fa_prefill_forward", "fa_forward_ws",
                                "fa_verify_forward"])
def test_argument_validation_returns_before_any_cuda_call(capi, fn):
    sq = 5 if fn == "fa_verify_forward" else 256
    assert call(capi, fn, q=None, Sq=sq) == capi.FA_ERR_INVALID_ARG
    assert call(capi, fn, lse=None, Sq=sq) == capi.FA_ERR_INVALID_ARG
    assert call(capi, fn, B=0, Sq=sq) == capi.FA_ERR_INVALID_ARG
    assert call(capi, fn, Sk=-1, Sq=sq) == capi.FA_ERR_INVALID_ARG
    assert call(capi, fn, scale=float("nan"), Sq=sq) == capi.FA_ERR_INVALID_ARG
    assert call(capi, fn, scale=float("inf"), Sq=sq) == capi.FA_ERR_INVALID_ARG
    assert call(capi, fn, d=96, Sq=sq) == capi.FA_ERR_UNSUPPORTED
    assert call(capi, fn, d=256, Sq=sq) == capi.FA_ERR_UNSUPPORTED
    assert call(capi, fn, q=ALIGNED + 8, Sq=sq) == capi.FA_ERR_UNSUPPORTED
    assert call(capi, fn, o=ALIGNED + 2, Sq=sq) == capi.FA_ERR_UNSUPPORTED
    assert call(capi, fn, lse=ALIGNED + 2, Sq=sq) == capi.FA_ERR_UNSUPPORTED
    assert call(capi, fn, Sq=sq, Sk=2**31) == capi.FA_ERR_UNSUPPORTED


def _no_device():
    import torch
    return not torch.cuda.is_available()


@pytest.mark.parametrize("fn", ["fa_forward", "fa_prefill_forward", "fa_forward_ws",
                                "fa_verify_forward"])
@pytest.mark.parametrize("scale", [0.0, -0.0, -0.5, -1e30, 3e-39])
def test_every_finite_scale_passes_validation(capi, fn, scale):
    """The pages make the scale a plain factor of the scores, so zero and
    negative values are valid. With no CUDA device the call gets past argument
    validation and fails only at the device lookup (FA_ERR_CUDA). The fake
    pointers must never reach a kernel, so this runs only where no device is
    visible."""
    if not _no_device():
        pytest.skip("fake pointers: only meaningful on a host without a CUDA device")
    sq = 5 if fn == "fa_verify_forward" else 256
    assert call(capi, fn, scale=scale, Sq=sq) == capi.FA_ERR_CUDA


def test_static_entry_checks_arguments_like_the_allocating_one(capi):
    """fa_verify_forward_static runs fa_verify_forward's checks, with the same
    codes, before its scratch-size check and before touching a device."""
    A = ALIGNED
    for f in (lambda *a: capi.fa_verify_forward_static(*a, 0),
              lambda *a: capi.fa_verify_forward(*a, None, 0, 0)):
        assert f(A, A, A, A, A, 1, 1, 17, 100, 128, 1, 0.1, 0) == capi.FA_ERR_UNSUPPORTED
        assert f(A, A, A, A, A, 256, 256, 5, 100, 128, 1, 0.1, 0) == capi.FA_ERR_UNSUPPORTED
        assert f(A, A, A, A, A, 1, 1, 5, 100, 128, 1, 0.1, 3) == capi.FA_ERR_INVALID_ARG
        assert f(A, A, A, A, A, 1, 1, 5, 100, 128, 1, 0.1, -1) == capi.FA_ERR_INVALID_ARG
        assert f(None, A, A, A, A, 1, 1, 5, 100, 128, 1, 0.1, 0) == capi.FA_ERR_INVALID_ARG
        assert f(A, A, A, A, A, 1, 1, 5, 100, 96, 1, 0.1, 0) == capi.FA_ERR_UNSUPPORTED
    # an explicit split count whose partials exceed the array: refused without a device
    assert capi.fa_verify_forward_static(A, A, A, A, A, 16, 32, 16, 4096, 128, 1, 0.1, 8, 0) == \
        capi.FA_ERR_WORKSPACE


def test_verify_specific_checks(capi):
    assert call(capi, "fa_verify_forward", Sq=17) == capi.FA_ERR_UNSUPPORTED
    assert call(capi, "fa_verify_forward", Sq=5, Sk=4096, n_split=-1) == capi.FA_ERR_INVALID_ARG
    assert call(capi, "fa_verify_forward", Sq=5, Sk=4096, n_split=65) == capi.FA_ERR_INVALID_ARG
    assert call(capi, "fa_verify_forward", Sq=5, B=256, H=256) == capi.FA_ERR_UNSUPPORTED


def test_workspace_size_is_zero_for_the_prefill_path(capi):
    assert capi.fa_workspace_size(4, 32, 8192, 8192, 128) == 0
    assert capi.fa_workspace_size(0, 32, 5, 4096, 128) == 0
    assert capi.fa_verify_workspace_size(16, 32, 5, 4096, 128, 1) == 0
    # explicit split counts need no device: fp32 partial O then LSE, each 256-byte aligned
    n = capi.fa_verify_workspace_size(16, 32, 5, 4096, 128, 4)
    o_bytes = 4 * 16 * 32 * 5 * 128 * 4
    l_bytes = -(-(4 * 16 * 32 * 5 * 4) // 256) * 256
    assert n == o_bytes + l_bytes


def test_tree_and_paged_entry_points_validate_first(capi):
    A = ALIGNED
    t = capi.fa_verify_tree_forward
    assert t(A, A, A, A, A, 1, 1, 5, 100, 128, None, 0.1, 0, None, 0, 0) == capi.FA_ERR_INVALID_ARG
    assert t(A, A, A, A, A, 1, 1, 5, 100, 128, A + 2, 0.1, 0, None, 0, 0) == capi.FA_ERR_INVALID_ARG
    assert t(A, A, A, A, A, 1, 1, 17, 100, 128, A, 0.1, 0, None, 0, 0) == capi.FA_ERR_UNSUPPORTED
    p = capi.fa_verify_paged_forward
    ok = dict(B=2, H=2, Sq=5, d=128, num_pages=10, page_size=16, max_pages=8, max_len=100)
    def call(**kw):
        a = dict(ok, **kw)
        return p(A, A, A, kw.get("table", A), kw.get("lens", A), A, A, a["B"], a["H"], a["Sq"],
                 a["d"], a["num_pages"], a["page_size"], a["max_pages"], a["max_len"], 1, None,
                 0.1, 0, None, 0, 0)
    assert call(table=None) == capi.FA_ERR_INVALID_ARG
    assert call(lens=None) == capi.FA_ERR_INVALID_ARG
    assert call(page_size=24) == capi.FA_ERR_UNSUPPORTED
    assert call(page_size=96) == capi.FA_ERR_UNSUPPORTED
    assert call(max_len=129) == capi.FA_ERR_INVALID_ARG     # > max_pages * page_size
    assert call(num_pages=0) == capi.FA_ERR_INVALID_ARG
    assert call(Sq=17) == capi.FA_ERR_UNSUPPORTED
    assert call(d=96) == capi.FA_ERR_UNSUPPORTED


def test_host_entry_point_validates_first(capi):
    f = capi.fa_forward_host
    assert f(None, 1, 1, 1, 1, 1, 1, 256, 256, 128, 1, 0.1, None, 0, 0) == capi.FA_ERR_INVALID_ARG
    assert f(1, 1, 1, 1, 1, 0, 1, 256, 256, 128, 1, 0.1, None, 0, 0) == capi.FA_ERR_INVALID_ARG
    assert f(1, 1, 1, 1, 1, 1, 1, 256, 256, 96, 1, 0.1, None, 0, 0) == capi.FA_ERR_UNSUPPORTED
    if _no_device():  # a negative scale is valid: only the device lookup fails
        assert f(1, 1, 1, 1, 1, 1, 1, 256, 256, 128, 1, -1.0, None, 0, 0) == capi.FA_ERR_CUDA
    assert capi.fa_forward_host_workspace_size(0, 1, 1, 1, 64) == 0


def test_testing_entry_points_validate_first(capi):
    assert capi.fa_selftest_umma(None, ALIGNED, ALIGNED, 128, 128, 0, 0) == capi.FA_ERR_INVALID_ARG
    assert capi.fa_selftest_umma(ALIGNED, ALIGNED, ALIGNED, 96, 128, 0, 0) == capi.FA_ERR_INVALID_ARG
    assert capi.fa_selftest_wait_timeout(0, 0) == capi.FA_ERR_INVALID_ARG
    assert capi.fa_selftest_elect(None, 4, 0) == capi.FA_ERR_INVALID_ARG
    assert capi.fa_selftest_elect(ALIGNED, 0, 0) == capi.FA_ERR_INVALID_ARG
    assert capi.fa_reference_forward_simt(None, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 1, 1, 4, 4, 8,
                                          0, 0.5, 0) == capi.FA_ERR_INVALID_ARG


def test_python_binding_refuses_a_missing_library(tmp_path):
    from exact_tiled_attention_03_gb300 import _capi
    saved = _capi._lib
    try:
        _capi._lib = None
        with pytest.raises(RuntimeError, match="no CPU fallback"):
            _capi.load(str(tmp_path / "nope.so"))
    finally:
        _capi._lib = saved
