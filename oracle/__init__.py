"""fp64 CPU oracle for the exact attention forward pass.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package. It
shares no code with the CUDA path and nothing in the product path calls it.

``oracle.c`` holds the arithmetic (the materialising two-pass definition, the
two online forms and the split-KV combine, each citing its passage);
``numpy_ref.py`` is an independent vectorised restatement of the definition
used only to cross-check the C code on small inputs. This file only marshals
arguments through ctypes.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the mutation tests load a copy of the oracle with a
        # planted mistake; nothing else sets it.
        path = os.environ.get("ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64p = ctypes.POINTER(ctypes.c_int64)
        dblp = ctypes.POINTER(ctypes.c_double)
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        common = [u16p, u16p, u16p, i64, i64, i64, i64, i64, i32, f32]
        L.oracle_attention_rows.argtypes = common + [i64p, i64, dblp, dblp, i32]
        L.oracle_attention.argtypes = common + [dblp, dblp, i32]
        L.oracle_probs_row.argtypes = [u16p, u16p, i64, i64, i64, i64, i64, i32, f32,
                                       i64, i64, i64, dblp]
        L.oracle_online_rows.argtypes = common + [i64, i32, i64p, i64, dblp, dblp, i32]
        L.oracle_split_rows.argtypes = common + [i64p, i64, i64p, i64, dblp, dblp, i32]
        L.oracle_combine.argtypes = [i64, i64, i64, dblp, dblp, dblp, dblp]
        L.oracle_attention_backward.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, i64, i64,
                                                i32, f32, dblp, dblp, dblp, i32]
        L.oracle_attention_backward_rows.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, i64,
                                                     i64, i32, f32, i64, i64p, i64, i64p, i64,
                                                     dblp, dblp, dblp, i32]
        L.oracle_attention_masked.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64, i64,
                                              ctypes.POINTER(ctypes.c_uint8), f32, dblp, dblp, i32]
        L.oracle_max_threads.argtypes = []
        u8p = ctypes.POINTER(ctypes.c_uint8)
        fp8 = [u8p, u8p, u8p, i64, i64, i64, i64, i64, i32, f32, f32, f32, f32, i32]
        L.oracle_attention_fp8_rows.argtypes = fp8 + [i64p, i64, dblp, dblp, i32]
        L.oracle_attention_fp8.argtypes = fp8 + [dblp, dblp, i32]
        L.oracle_e4m3_decode.argtypes = [u8p, i64, dblp]
        L.oracle_e4m3_round.argtypes = [dblp, i64, dblp]
        for f in (L.oracle_attention_rows, L.oracle_attention, L.oracle_probs_row,
                  L.oracle_online_rows, L.oracle_split_rows, L.oracle_max_threads,
                  L.oracle_combine, L.oracle_attention_masked, L.oracle_attention_backward,
                  L.oracle_attention_backward_rows, L.oracle_attention_fp8_rows,
                  L.oracle_attention_fp8, L.oracle_e4m3_decode, L.oracle_e4m3_round):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _bits(t: torch.Tensor) -> np.ndarray:
    """bf16 CPU tensor -> contiguous uint16 array of its bit patterns."""
    if t.dtype != torch.bfloat16:
        raise TypeError(f"oracle inputs are bf16, got {t.dtype}")
    t = t.detach().to("cpu").contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _dims(q, k, v):
    if q.dim() != 4 or k.shape != v.shape or k.dim() != 4:
        raise ValueError("expected q [B,H,Sq,d] and k, v [B,H,Sk,d]")
    B, H, Sq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("q and k/v disagree on B, H or d")
    return B, H, Sq, k.shape[2], d


def _rows_array(rows, B, H, Sq):
    if rows is None:
        return None
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    return r


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def attention(q, k, v, causal: bool, scale: float, rows=None, threads: int = 0):
    """Definition of attention in fp64.

    rows=None: returns (o [B,H,Sq,d], lse [B,H,Sq]) float64 arrays.
    rows=[(b,h,i), ...]: returns (o [n,d], lse [n]) for those rows.
    """
    B, H, Sq, Sk, d = _dims(q, k, v)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    L = lib()
    args = (_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
            B, H, Sq, Sk, d, int(bool(causal)), ctypes.c_float(scale))
    if rows is None:
        o = np.empty((B, H, Sq, d), dtype=np.float64)
        lse = np.empty((B, H, Sq), dtype=np.float64)
        _check(L.oracle_attention(*args, _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                  int(threads)), "attention")
        return o, lse
    r = _rows_array(rows, B, H, Sq)
    n = r.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _check(L.oracle_attention_rows(*args, _ptr(r, ctypes.c_int64), n, _ptr(o, ctypes.c_double),
                                   _ptr(lse, ctypes.c_double), int(threads)), "attention_rows")
    return o, lse


def probs_row(q, k, causal: bool, scale: float, b: int, h: int, i: int):
    """Softmax row P_i over all Sk keys (hidden keys 0), fp64."""
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    qb, kb = _bits(q), _bits(k)
    p = np.empty((Sk,), dtype=np.float64)
    _check(lib().oracle_probs_row(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), B, H, Sq,
                                  Sk, d, int(bool(causal)), ctypes.c_float(scale), b, h, i,
                                  _ptr(p, ctypes.c_double)), "probs_row")
    return p


def _all_rows(B, H, Sq):
    return [(b, h, i) for b in range(B) for h in range(H) for i in range(Sq)]


def online(q, k, v, causal: bool, scale: float, block: int, form: int, rows=None, threads=0):
    """Online (block-wise, one-pass) softmax forms; form 1 = page 1, form 2 = page 2 Ch. 3."""
    B, H, Sq, Sk, d = _dims(q, k, v)
    r = _rows_array(rows if rows is not None else _all_rows(B, H, Sq), B, H, Sq)
    n = r.shape[0]
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _check(lib().oracle_online_rows(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                    _ptr(vb, ctypes.c_uint16), B, H, Sq, Sk, d,
                                    int(bool(causal)), ctypes.c_float(scale), int(block), int(form),
                                    _ptr(r, ctypes.c_int64), n, _ptr(o, ctypes.c_double),
                                    _ptr(lse, ctypes.c_double), int(threads)), "online_rows")
    return o, lse


def split(q, k, v, causal: bool, scale: float, bounds, rows=None, threads=0):
    """Split-KV partials over key chunks cut at ``bounds`` plus the final LSE combine."""
    B, H, Sq, Sk, d = _dims(q, k, v)
    r = _rows_array(rows if rows is not None else _all_rows(B, H, Sq), B, H, Sq)
    n = r.shape[0]
    bnd = np.ascontiguousarray(np.asarray(bounds, dtype=np.int64))
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _check(lib().oracle_split_rows(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                   _ptr(vb, ctypes.c_uint16), B, H, Sq, Sk, d, int(bool(causal)),
                                   ctypes.c_float(scale), _ptr(bnd, ctypes.c_int64),
                                   len(bnd) - 1, _ptr(r, ctypes.c_int64), n,
                                   _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                   int(threads)), "split_rows")
    return o, lse


def combine(o_parts, lse_parts):
    """Combine per-part (o, lse) computed elsewhere: o_parts [P, n, d], lse_parts [P, n]."""
    op = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    lp = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    P, n, d = op.shape
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _check(lib().oracle_combine(P, n, d, _ptr(op, ctypes.c_double), _ptr(lp, ctypes.c_double),
                                _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double)), "combine")
    return o, lse


def attention_masked(q, k, v, visible, scale: float, threads: int = 0):
    """Definition with an explicit mask: visible [B, Sq, Sk] (nonzero = key enters the row)."""
    B, H, Sq, Sk, d = _dims(q, k, v)
    vis = np.ascontiguousarray(np.asarray(visible, dtype=np.uint8).reshape(B, Sq, Sk))
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    o = np.empty((B, H, Sq, d), dtype=np.float64)
    lse = np.empty((B, H, Sq), dtype=np.float64)
    _check(lib().oracle_attention_masked(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                         _ptr(vb, ctypes.c_uint16), B, H, Sq, Sk, d,
                                         _ptr(vis, ctypes.c_uint8), ctypes.c_float(scale),
                                         _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                         int(threads)), "attention_masked")
    return o, lse


def attention_backward(q, k, v, dout, causal: bool, scale: float, threads: int = 0):
    """Gradients (dq, dk, dv) of the definition for upstream gradient dout, fp64."""
    B, H, Sq, Sk, d = _dims(q, k, v)
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    dq = np.empty((B, H, Sq, d), dtype=np.float64)
    dk = np.empty((B, H, Sk, d), dtype=np.float64)
    dv = np.empty((B, H, Sk, d), dtype=np.float64)
    _check(lib().oracle_attention_backward(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                           _ptr(vb, ctypes.c_uint16), _ptr(db, ctypes.c_uint16),
                                           B, H, Sq, Sk, d, int(bool(causal)),
                                           ctypes.c_float(scale), _ptr(dq, ctypes.c_double),
                                           _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
                                           int(threads)), "attention_backward")
    return dq, dk, dv


def attention_backward_rows(q, k, v, dout, causal: bool, scale: float, b: int, h: int, qrows,
                            krows, threads: int = 0):
    """dQ of the chosen query rows and dK, dV of the chosen key rows of head (b, h)."""
    B, H, Sq, Sk, d = _dims(q, k, v)
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int64))
    kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int64))
    dq = np.empty((len(qr), d), dtype=np.float64)
    dk = np.empty((len(kr), d), dtype=np.float64)
    dv = np.empty((len(kr), d), dtype=np.float64)
    _check(lib().oracle_attention_backward_rows(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        _ptr(db, ctypes.c_uint16), B, H, Sq, Sk, d, int(bool(causal)), ctypes.c_float(scale),
        b * H + h, _ptr(qr, ctypes.c_int64), len(qr), _ptr(kr, ctypes.c_int64), len(kr),
        _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
        int(threads)), "attention_backward_rows")
    return dq, dk, dv


def _bytes(t: torch.Tensor) -> np.ndarray:
    """E4M3 tensor (torch.float8_e4m3fn) or uint8 bytes -> contiguous uint8 array."""
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"FP8 oracle inputs are E4M3 bytes, got {t.dtype}")
    return t.detach().to("cpu").contiguous().numpy()


def e4m3_decode(x) -> np.ndarray:
    """Exact value of each E4M3 byte (NaN for the NaN codes), fp64."""
    b = np.ascontiguousarray(np.asarray(x, dtype=np.uint8)).reshape(-1)
    out = np.empty(b.shape, dtype=np.float64)
    _check(lib().oracle_e4m3_decode(_ptr(b, ctypes.c_uint8), b.size, _ptr(out, ctypes.c_double)),
           "e4m3_decode")
    return out


def e4m3_round(y) -> np.ndarray:
    """Nearest E4M3 value (ties to even, |y| > 448 clamped), fp64."""
    a = np.ascontiguousarray(np.asarray(y, dtype=np.float64)).reshape(-1)
    out = np.empty(a.shape, dtype=np.float64)
    _check(lib().oracle_e4m3_round(_ptr(a, ctypes.c_double), a.size, _ptr(out, ctypes.c_double)),
           "e4m3_round")
    return out


def attention_fp8(q8, k8, v8, causal: bool, scale: float, descale=(1.0, 1.0, 1.0),
                  quantize_p: bool = True, rows=None, threads: int = 0):
    """FP8 forward: E4M3 inputs times per-tensor descales, P rounded to E4M3 when
    ``quantize_p`` (else the definition on the decoded inputs). Shapes and return
    values as ``attention``."""
    if q8.dim() != 4 or k8.shape != v8.shape or k8.dim() != 4:
        raise ValueError("expected q [B,H,Sq,d] and k, v [B,H,Sk,d]")
    B, H, Sq, d = q8.shape
    Sk = k8.shape[2]
    qb, kb, vb = _bytes(q8), _bytes(k8), _bytes(v8)
    L = lib()
    args = (_ptr(qb, ctypes.c_uint8), _ptr(kb, ctypes.c_uint8), _ptr(vb, ctypes.c_uint8),
            B, H, Sq, Sk, d, int(bool(causal)), ctypes.c_float(scale),
            ctypes.c_float(descale[0]), ctypes.c_float(descale[1]), ctypes.c_float(descale[2]),
            int(bool(quantize_p)))
    if rows is None:
        o = np.empty((B, H, Sq, d), dtype=np.float64)
        lse = np.empty((B, H, Sq), dtype=np.float64)
        _check(L.oracle_attention_fp8(*args, _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                      int(threads)), "attention_fp8")
        return o, lse
    r = _rows_array(rows, B, H, Sq)
    n = r.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _check(L.oracle_attention_fp8_rows(*args, _ptr(r, ctypes.c_int64), n,
                                       _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                       int(threads)), "attention_fp8_rows")
    return o, lse


__all__ = ["attention", "attention_backward", "attention_backward_rows", "attention_masked",
           "attention_fp8", "e4m3_decode", "e4m3_round", "probs_row", "online", "split",
           "combine", "max_threads", "lib"]
