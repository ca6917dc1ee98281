"""ctypes binding of the C ABI in include/fa.h and include/fa_testing.h.

Argument marshalling only: every entry point keeps its C name and argument
order; a torch tensor may stand wherever the C call takes a device pointer,
and a torch.cuda.Stream (or None = torch's current stream) where it takes a
stream. There is no fallback: if the CUDA library is missing the first call
raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_WORKSPACE = 5
FA_ERR_BOUNDS = 6
FA_VERIFY_MAX_SQ = 16
FA_STATIC_SCRATCH_BYTES = 8 * 1024 * 1024
FA_HOST_CHUNKS = 16

# Every function the headers declare, with its ctypes signature.
_P, _I64, _I32, _F32, _SZ, _U64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                   ctypes.c_size_t, ctypes.c_uint64)
_ATTN = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I32, _F32]
SIGNATURES = {
    "fa_forward": (_I32, _ATTN + [_P]),
    "fa_workspace_size": (_SZ, [_I64] * 5),
    "fa_forward_ws": (_I32, _ATTN + [_P, _SZ, _P]),
    "fa_prefill_forward": (_I32, _ATTN + [_P]),
    "fa_forward_fp8": (_I32, _ATTN + [_F32, _F32, _F32, _P]),
    "fa_verify_forward": (_I32, _ATTN + [_I32, _P, _SZ, _P]),
    "fa_verify_workspace_size": (_SZ, [_I64] * 5 + [_I32]),
    "fa_verify_auto_splits": (_I32, [_I64] * 5),
    "fa_verify_forward_static": (_I32, _ATTN + [_I32, _P]),
    "fa_forward_host": (_I32, _ATTN + [_P, _SZ, _P]),
    "fa_backward": (_I32, [_P] * 9 + [_I64] * 5 + [_I32, _F32, _P, _SZ, _P]),
    "fa_backward_workspace_size": (_SZ, [_I64] * 5),
    "fa_verify_tree_forward": (_I32, [_P] * 5 + [_I64] * 5 + [_P, _F32, _I32, _P, _SZ, _P]),
    "fa_verify_paged_forward": (_I32, [_P] * 7 + [_I64] * 8 + [_I32, _P, _F32, _I32, _P, _SZ, _P]),
    "fa_forward_host_workspace_size": (_SZ, [_I64] * 5),
    "fa_status_string": (ctypes.c_char_p, [_I32]),
    "fa_device_status": (_I32, [_P]),
    "fa_reference_forward_simt": (_I32, _ATTN + [_P]),
    "fa_selftest_umma": (_I32, [_P, _P, _P, _I32, _I32, _I32, _P]),
    "fa_selftest_umma_ts": (_I32, [_P, _P, _P, _I32, _I32, _I32, _P]),
    "fa_selftest_umma_f8": (_I32, [_P, _P, _P, _I32, _I32, _I32, _P]),
    "fa_selftest_wait_timeout": (_I32, [_U64, _P]),
    "fa_testing_stall_next_launch": (_I32, [_I32, _I32, _U64]),
    "fa_testing_debug_checks": (_I32, []),
    "fa_selftest_index_check": (_I32, [_I32, _P]),
    "fa_selftest_elect": (_I32, [_P, _I32, _P]),
    "fa_selftest_mufu": (_I32, [_P, _I32, _I32, _P]),
    "fa_selftest_mma_rate": (_I32, [_P, _I32, _I32, _I32, _P]),
}

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def open_library(path: str):
    """A handle on a build of the library at `path` (for example the debug build),
    with every signature set; it does not become the handle the wrappers use."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"the CUDA library {path} is missing; build it with "
            "`python -m exact_tiled_attention_03_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


def load(path: str | None = None):
    """Load the CUDA library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = open_library(path or LIB_PATH)
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a tensor, an int address or None, got {type(x).__name__}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_status_string(status: int) -> str:
    return status_string(status)


def fa_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream=None) -> int:
    return load().fa_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk, d,
                             int(bool(causal)), float(scale), _stream(stream))


def fa_workspace_size(B, H, Sq, Sk, d) -> int:
    return load().fa_workspace_size(B, H, Sq, Sk, d)


def fa_forward_ws(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, workspace, ws_bytes,
                  stream=None) -> int:
    return load().fa_forward_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk, d,
                                int(bool(causal)), float(scale), _ptr(workspace), int(ws_bytes),
                                _stream(stream))


def fa_prefill_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, stream=None) -> int:
    return load().fa_prefill_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk,
                                     d, int(bool(causal)), float(scale), _stream(stream))


def fa_forward_fp8(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, q_descale, k_descale,
                   v_descale, stream=None) -> int:
    return load().fa_forward_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk, d,
                                 int(bool(causal)), float(scale), float(q_descale),
                                 float(k_descale), float(v_descale), _stream(stream))


def fa_verify_forward(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, n_split, workspace,
                      ws_bytes, stream=None) -> int:
    return load().fa_verify_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk,
                                    d, int(bool(causal)), float(scale), int(n_split),
                                    _ptr(workspace), int(ws_bytes), _stream(stream))


def fa_verify_forward_static(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, n_split,
                             stream=None) -> int:
    return load().fa_verify_forward_static(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                           Sq, Sk, d, int(bool(causal)), float(scale),
                                           int(n_split), _stream(stream))


def fa_verify_tree_forward(q, k, v, o, lse, B, H, Sq, Sk, d, tree_mask, scale, n_split, workspace,
                           ws_bytes, stream=None) -> int:
    return load().fa_verify_tree_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq,
                                         Sk, d, _ptr(tree_mask), float(scale), int(n_split),
                                         _ptr(workspace), int(ws_bytes), _stream(stream))


def fa_verify_paged_forward(q, k_pages, v_pages, block_table, seq_lens, o, lse, B, H, Sq, d,
                            num_pages, page_size, max_pages_per_seq, max_seq_len, causal,
                            tree_mask, scale, n_split, workspace, ws_bytes, stream=None) -> int:
    return load().fa_verify_paged_forward(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens), _ptr(o),
        _ptr(lse), B, H, Sq, d, num_pages, page_size, max_pages_per_seq, max_seq_len,
        int(bool(causal)), _ptr(tree_mask), float(scale), int(n_split), _ptr(workspace),
        int(ws_bytes), _stream(stream))


def fa_backward(q, k, v, o, lse, dout, dq, dk, dv, B, H, Sq, Sk, d, causal, scale, workspace=None,
                ws_bytes=0, stream=None) -> int:
    return load().fa_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, H, Sq, Sk, d, int(bool(causal)),
                              float(scale), _ptr(workspace), int(ws_bytes), _stream(stream))


def fa_backward_workspace_size(B, H, Sq, Sk, d) -> int:
    return load().fa_backward_workspace_size(B, H, Sq, Sk, d)


def fa_forward_host(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale, workspace=None, ws_bytes=0,
                    stream=None) -> int:
    return load().fa_forward_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk, d,
                                  int(bool(causal)), float(scale), _ptr(workspace), int(ws_bytes),
                                  _stream(stream))


def fa_forward_host_workspace_size(B, H, Sq, Sk, d) -> int:
    return load().fa_forward_host_workspace_size(B, H, Sq, Sk, d)


def fa_verify_workspace_size(B, H, Sq, Sk, d, n_split) -> int:
    return load().fa_verify_workspace_size(B, H, Sq, Sk, d, int(n_split))


def fa_verify_auto_splits(B, H, Sq, Sk, d) -> int:
    return load().fa_verify_auto_splits(B, H, Sq, Sk, d)


def fa_device_status(stream=None) -> int:
    return load().fa_device_status(_stream(stream))


def fa_reference_forward_simt(q, k, v, o, lse, B, H, Sq, Sk, d, causal, scale,
                              stream=None) -> int:
    return load().fa_reference_forward_simt(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                            Sq, Sk, d, int(bool(causal)), float(scale),
                                            _stream(stream))


def fa_selftest_umma(a, b, c, n, k, b_mn_major, stream=None) -> int:
    return load().fa_selftest_umma(_ptr(a), _ptr(b), _ptr(c), int(n), int(k), int(b_mn_major),
                                   _stream(stream))


def fa_selftest_umma_ts(a, b, c, n, k, b_mn_major, stream=None) -> int:
    return load().fa_selftest_umma_ts(_ptr(a), _ptr(b), _ptr(c), int(n), int(k), int(b_mn_major),
                                      _stream(stream))


def fa_selftest_umma_f8(a, b, c, n, b_mn_major, a_tmem, stream=None) -> int:
    return load().fa_selftest_umma_f8(_ptr(a), _ptr(b), _ptr(c), int(n), int(b_mn_major),
                                      int(a_tmem), _stream(stream))


def fa_selftest_mufu(out, blocks, iters, stream=None) -> int:
    return load().fa_selftest_mufu(_ptr(out), int(blocks), int(iters), _stream(stream))


def fa_selftest_mma_rate(cycles, mode, blocks, iters, stream=None) -> int:
    return load().fa_selftest_mma_rate(_ptr(cycles), int(mode), int(blocks), int(iters),
                                       _stream(stream))


def fa_selftest_wait_timeout(timeout_ns, stream=None) -> int:
    return load().fa_selftest_wait_timeout(int(timeout_ns), _stream(stream))


def fa_testing_stall_next_launch(kernel, skip_index, wait_limit_ns) -> int:
    return load().fa_testing_stall_next_launch(int(kernel), int(skip_index), int(wait_limit_ns))


STALL_PREFILL = 1
STALL_VERIFY = 2


def check(status: int, what: str = "fa call"):
    if status != FA_OK:
        raise FAError(status, what)


def fa_testing_debug_checks() -> int:
    return load().fa_testing_debug_checks()


def fa_selftest_index_check(fail, stream=None) -> int:
    return load().fa_selftest_index_check(int(bool(fail)), _stream(stream))


def fa_selftest_elect(lanes, trials, stream=None) -> int:
    return load().fa_selftest_elect(_ptr(lanes), int(trials), _stream(stream))
