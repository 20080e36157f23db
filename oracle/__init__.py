"""FP64 CPU oracle for fused causal attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  It shares nothing with the CUDA library: the
arithmetic lives in ``attn_oracle.c`` (plain C, FP64) and this module only
marshals numpy arrays into it.

What it computes (TransformerEngine PR #3527, "cuDNN FROST attention backend",
description and review notes; PR #3699 for keyless rows):

* ``fwd``: O = softmax(scale * Q K^T + mask) V per (sequence, query head) and the
  natural-log LSE, in float64; rows with no visible key give O = 0, LSE = -inf.
* ``bwd``: the exact gradients dQ, dK, dV of O for an upstream dO, with the
  oracle's own FP64 O (D_i = dO_i . O_i).
* ``lse_merge``: the LSE-weighted combination of partial results over disjoint
  key sets, as a context-parallel ring uses it.
* ``naive``: the unfused reduced-precision implementation whose error against
  ``fwd``/``bwd`` is the accuracy floor of the 2x criterion.
* ``bwd_kv`` / ``naive_kv``: ``bwd``'s and ``naive``'s dK, dV restricted to
  selected key rows (every query row that sees one still gets its complete
  forward), for checking deep accumulations of full-size problems.

Every function is pinned by ``tests/test_oracle_pins.py`` against things other
than itself: torch's float64 attention and autograd (library routines), central
finite differences, closed forms and invariants.

Layout: THD throughout -- q [Tq, hq, dqk], k [Tk, hkv, dqk], v [Tk, hkv, dv],
o/dout [Tq, hq, dv], lse [hq, Tq]; sequence b is rows [cu[b], cu[b+1]).
A dense [B, S, H, d] tensor is the same memory with cu = [0, S, 2S, ...].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libattn_oracle.so")
_lib = None
_lock = threading.Lock()

BF16, FP16, FP32 = 0, 1, 2
_DTYPE_CODES = {"bf16": BF16, "bfloat16": BF16, "fp16": FP16, "float16": FP16,
                "fp32": FP32, "float32": FP32}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build`` (idempotent)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32p = ctypes.POINTER(ctypes.c_int32)
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        ci, cd = ctypes.c_int, ctypes.c_double
        lib.oracle_fwd.argtypes = [ci, i32p, i32p, ci, ci, ci, ci, dp, dp, dp,
                                   ci, ci, ci, ci, cd, dp, dp, u8p, ci]
        lib.oracle_fwd.restype = ci
        lib.oracle_bwd.argtypes = [ci, i32p, i32p, ci, ci, ci, ci, dp, dp, dp, dp,
                                   ci, ci, ci, ci, cd, dp, dp, dp, u8p, ci]
        lib.oracle_bwd.restype = ci
        lib.oracle_lse_merge.argtypes = [ci, ctypes.c_long, ci, ci, dp, dp, dp, dp]
        lib.oracle_lse_merge.restype = ci
        lib.oracle_naive.argtypes = [ci, i32p, i32p, ci, ci, ci, ci, fp, fp, fp, fp,
                                     ci, ci, ci, ci, cd, ci, fp, fp, fp, fp, fp, ci]
        lib.oracle_naive.restype = ci
        lib.oracle_bwd_kv.argtypes = [ci, i32p, i32p, ci, ci, ci, ci, dp, dp, dp, dp,
                                      ci, ci, ci, ci, cd, u8p, u8p, dp, dp, ci]
        lib.oracle_bwd_kv.restype = ci
        lib.oracle_naive_kv.argtypes = [ci, i32p, i32p, ci, ci, ci, ci, fp, fp, fp, fp,
                                        ci, ci, ci, ci, cd, ci, u8p, u8p, fp, fp, ci]
        lib.oracle_naive_kv.restype = ci
        _lib = lib
        return lib


def _nthreads(n):
    if n:
        return int(n)
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _cu(cu):
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int32))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle {name}: invalid arguments (code {rc})")


def fwd(q, k, v, cu_q, cu_k, *, scale, causal=True, bottom_right=False,
        window=(-1, -1), heads=None, nthreads=None):
    """Exact forward. Returns (o [Tq,hq,dv], lse [hq,Tq]) in float64.

    ``heads``: optional iterable of query heads to compute (others stay 0/NaN).
    """
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q, cu_k = _cu(cu_q), _cu(cu_k)
    tq, hq, dqk = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    o = np.zeros((tq, hq, dv))
    lse = np.full((hq, tq), np.nan)
    sel = None
    if heads is not None:
        sel = np.zeros(hq, np.uint8)
        sel[list(heads)] = 1
    rc = lib.oracle_fwd(len(cu_q) - 1, _ptr(cu_q, ctypes.c_int32), _ptr(cu_k, ctypes.c_int32),
                        hq, hkv, dqk, dv, _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                        _ptr(v, ctypes.c_double), int(causal), int(bottom_right),
                        int(window[0]), int(window[1]), float(scale),
                        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                        None if sel is None else _ptr(sel, ctypes.c_uint8), _nthreads(nthreads))
    _check(rc, "fwd")
    return o, lse


def bwd(q, k, v, dout, cu_q, cu_k, *, scale, causal=True, bottom_right=False,
        window=(-1, -1), groups=None, nthreads=None):
    """Exact backward. Returns (dq, dk, dv) in float64.

    ``groups``: optional iterable of key/value heads whose group to compute.
    """
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu_q, cu_k = _cu(cu_q), _cu(cu_k)
    tq, hq, dqk = q.shape
    tk, hkv, dv = v.shape
    dq = np.zeros_like(q)
    dk = np.zeros((tk, hkv, dqk))
    dvv = np.zeros((tk, hkv, dv))
    sel = None
    if groups is not None:
        sel = np.zeros(hkv, np.uint8)
        sel[list(groups)] = 1
    rc = lib.oracle_bwd(len(cu_q) - 1, _ptr(cu_q, ctypes.c_int32), _ptr(cu_k, ctypes.c_int32),
                        hq, hkv, dqk, dv, _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                        _ptr(v, ctypes.c_double), _ptr(dout, ctypes.c_double), int(causal),
                        int(bottom_right), int(window[0]), int(window[1]), float(scale),
                        _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                        _ptr(dvv, ctypes.c_double),
                        None if sel is None else _ptr(sel, ctypes.c_uint8), _nthreads(nthreads))
    _check(rc, "bwd")
    return dq, dk, dvv


def lse_merge(o_parts, lse_parts):
    """Merge partials: o_parts [n, rows, heads, dv], lse_parts [n, heads, rows]."""
    lib = _load()
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    n, rows, heads, dv = o_parts.shape
    assert lse_parts.shape == (n, heads, rows)
    o = np.zeros((rows, heads, dv))
    lse = np.zeros((heads, rows))
    rc = lib.oracle_lse_merge(n, rows, heads, dv, _ptr(o_parts, ctypes.c_double),
                              _ptr(lse_parts, ctypes.c_double), _ptr(o, ctypes.c_double),
                              _ptr(lse, ctypes.c_double))
    _check(rc, "lse_merge")
    return o, lse


def naive(q, k, v, cu_q, cu_k, *, scale, dtype="bf16", dout=None, causal=True,
          bottom_right=False, window=(-1, -1), nthreads=None):
    """Naive reduced-precision implementation (accuracy floor).

    Inputs must hold values representable in ``dtype``.  Returns
    (o, lse) or, with ``dout``, (o, lse, dq, dk, dv) as float32 arrays.
    """
    lib = _load()
    code = _DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    q, k, v = _f32(q), _f32(k), _f32(v)
    cu_q, cu_k = _cu(cu_q), _cu(cu_k)
    tq, hq, dqk = q.shape
    tk, hkv, dv = v.shape
    o = np.zeros((tq, hq, dv), np.float32)
    lse = np.zeros((hq, tq), np.float32)
    fptr = lambda a: _ptr(a, ctypes.c_float)  # noqa: E731
    if dout is not None:
        dout = _f32(dout)
        dq = np.zeros_like(q)
        dk = np.zeros((tk, hkv, dqk), np.float32)
        dvv = np.zeros((tk, hkv, dv), np.float32)
        args = (fptr(dout),)
        outs = (fptr(dq), fptr(dk), fptr(dvv))
    else:
        args = (None,)
        outs = (None, None, None)
    rc = lib.oracle_naive(len(cu_q) - 1, _ptr(cu_q, ctypes.c_int32), _ptr(cu_k, ctypes.c_int32),
                          hq, hkv, dqk, dv, fptr(q), fptr(k), fptr(v), *args, int(causal),
                          int(bottom_right), int(window[0]), int(window[1]), float(scale),
                          code, fptr(o), fptr(lse), *outs, _nthreads(nthreads))
    _check(rc, "naive")
    if dout is None:
        return o, lse
    return o, lse, dq, dk, dvv


def _key_sel(key_rows, tk):
    sel = np.zeros(tk, np.uint8)
    sel[np.asarray(list(key_rows), dtype=np.int64)] = 1
    return sel


def _group_sel(groups, hkv):
    if groups is None:
        return None
    sel = np.zeros(hkv, np.uint8)
    sel[list(groups)] = 1
    return sel


def bwd_kv(q, k, v, dout, cu_q, cu_k, *, scale, key_rows, causal=True, bottom_right=False,
           window=(-1, -1), groups=None, nthreads=None):
    """Exact dK, dV (float64) of the key rows ``key_rows`` (global rows of the
    packed K) and, optionally, only the key/value heads ``groups``; the other
    entries of the returned arrays are 0.  Same definition as ``bwd``."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu_q, cu_k = _cu(cu_q), _cu(cu_k)
    tq, hq, dqk = q.shape
    tk, hkv, dv = v.shape
    dk = np.zeros((tk, hkv, dqk))
    dvv = np.zeros((tk, hkv, dv))
    ks = _key_sel(key_rows, tk)
    gs = _group_sel(groups, hkv)
    rc = lib.oracle_bwd_kv(len(cu_q) - 1, _ptr(cu_q, ctypes.c_int32), _ptr(cu_k, ctypes.c_int32),
                           hq, hkv, dqk, dv, _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                           _ptr(v, ctypes.c_double), _ptr(dout, ctypes.c_double), int(causal),
                           int(bottom_right), int(window[0]), int(window[1]), float(scale),
                           _ptr(ks, ctypes.c_uint8),
                           None if gs is None else _ptr(gs, ctypes.c_uint8),
                           _ptr(dk, ctypes.c_double), _ptr(dvv, ctypes.c_double),
                           _nthreads(nthreads))
    _check(rc, "bwd_kv")
    return dk, dvv


def naive_kv(q, k, v, dout, cu_q, cu_k, *, scale, key_rows, dtype="bf16", causal=True,
             bottom_right=False, window=(-1, -1), groups=None, nthreads=None):
    """The naive implementation's dK, dV (float32) of the key rows ``key_rows``
    (and key/value heads ``groups``); other entries are 0.  Same arithmetic as
    ``naive`` except the order of the FP32 sums over query rows."""
    lib = _load()
    code = _DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    cu_q, cu_k = _cu(cu_q), _cu(cu_k)
    tq, hq, dqk = q.shape
    tk, hkv, dv = v.shape
    dk = np.zeros((tk, hkv, dqk), np.float32)
    dvv = np.zeros((tk, hkv, dv), np.float32)
    ks = _key_sel(key_rows, tk)
    gs = _group_sel(groups, hkv)
    fptr = lambda a: _ptr(a, ctypes.c_float)  # noqa: E731
    rc = lib.oracle_naive_kv(len(cu_q) - 1, _ptr(cu_q, ctypes.c_int32),
                             _ptr(cu_k, ctypes.c_int32), hq, hkv, dqk, dv, fptr(q), fptr(k),
                             fptr(v), fptr(dout), int(causal), int(bottom_right),
                             int(window[0]), int(window[1]), float(scale), code,
                             _ptr(ks, ctypes.c_uint8),
                             None if gs is None else _ptr(gs, ctypes.c_uint8),
                             fptr(dk), fptr(dvv), _nthreads(nthreads))
    _check(rc, "naive_kv")
    return dk, dvv


def dense_cu(batch, seqlen):
    """Sequence offsets that make a dense [B, S, ...] tensor a THD tensor."""
    return np.arange(batch + 1, dtype=np.int32) * int(seqlen)
