"""ctypes binding of libattn.so (see include/attn.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  There is no fallback: if the library is missing or a call fails, an
exception is raised.

Tensors:
  dense: q [B, Sq, Hq, dqk], k [B, Sk, Hkv, dqk], v [B, Sk, Hkv, dv] (any
         strides with a contiguous last dimension);
  THD:   q [Tq, Hq, dqk], ... with int32 ``cu_seqlens_q/k`` on the device.
LSE is float32 [B, Hq, Sq] (dense) or [Hq, Tq] (THD), natural log.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libattn.so")

BF16, FP16, FP32 = 0, 1, 2
_STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
           3: "ATTN_ERR_ALIGNMENT", 4: "ATTN_ERR_WORKSPACE", 5: "ATTN_ERR_BAD_METADATA",
           6: "ATTN_ERR_TIMEOUT", 7: "ATTN_ERR_CUDA"}
EXPORTED = ["attn_fwd_workspace_size", "attn_bwd_workspace_size", "attn_fwd", "attn_bwd",
            "attn_bwd_preprocess", "attn_bwd_dq", "attn_bwd_dkdv", "attn_bwd_noalloc",
            "attn_lse_merge", "attn_cp_relayout",
            "attn_query_status", "attn_last_error", "attn_last_launch_count",
            "attn_debug_inject", "attn_host_arena_size", "attn_fwd_bwd_host",
            "attn_fwd_bwd_host_stages", "attn_bwd_path"]
# attn_fwd_bwd_host_stages stage bits
HOST_UPLOAD, HOST_COMPUTE, HOST_DOWNLOAD, HOST_ALL = 1, 2, 4, 7
# attn_bwd_path results: which backward kernels run (and the stage order)
BWD_RECOMPUTE, BWD_DS, BWD_PDS = 0, 1, 2
# attn_debug_inject kernel bits (test only)
DEBUG_FWD, DEBUG_DQ, DEBUG_DKDV, DEBUG_SCORES = 1, 2, 4, 8


class AttnError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{_STATUS.get(code, code)}: {msg}")
        self.code = code


class Params(ctypes.Structure):
    """Mirror of attn_params_t."""
    _fields_ = [
        ("dtype", ctypes.c_int), ("o_dtype", ctypes.c_int), ("grad_dtype", ctypes.c_int),
        ("batch", ctypes.c_int), ("seqlen_q", ctypes.c_int), ("seqlen_k", ctypes.c_int),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("total_q", ctypes.c_int), ("total_k", ctypes.c_int),
        ("heads_q", ctypes.c_int), ("heads_kv", ctypes.c_int),
        ("d_qk", ctypes.c_int), ("d_v", ctypes.c_int),
        ("stride_q", ctypes.c_int64 * 3), ("stride_k", ctypes.c_int64 * 3),
        ("stride_v", ctypes.c_int64 * 3), ("stride_o", ctypes.c_int64 * 3),
        ("stride_do", ctypes.c_int64 * 3), ("stride_dq", ctypes.c_int64 * 3),
        ("stride_dk", ctypes.c_int64 * 3), ("stride_dv", ctypes.c_int64 * 3),
        ("stride_lse", ctypes.c_int64 * 2),
        ("causal", ctypes.c_int), ("bottom_right", ctypes.c_int),
        ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("accumulate", ctypes.c_int),
        ("seqused_q", ctypes.c_void_p), ("seqused_k", ctypes.c_void_p),
        ("bwd_ds", ctypes.c_int),
    ]


_lib = None
_lock = threading.Lock()


def load():
    """Load libattn.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "bwd_tcgen05_tmem_gb300.build.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(Params)
        vp, sz, i64p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int64)
        lib.attn_fwd_workspace_size.argtypes = [P]
        lib.attn_fwd_workspace_size.restype = sz
        lib.attn_bwd_workspace_size.argtypes = [P]
        lib.attn_bwd_workspace_size.restype = sz
        lib.attn_bwd_path.argtypes = [P]
        lib.attn_bwd_path.restype = ctypes.c_int
        lib.attn_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.attn_fwd.restype = ctypes.c_int
        for name in ("attn_bwd", "attn_bwd_preprocess", "attn_bwd_dq", "attn_bwd_dkdv"):
            fn = getattr(lib, name)
            fn.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            fn.restype = ctypes.c_int
        lib.attn_bwd_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.attn_bwd_noalloc.restype = ctypes.c_int
        lib.attn_lse_merge.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                       i64p, i64p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       vp, ctypes.c_int, vp, vp]
        lib.attn_lse_merge.restype = ctypes.c_int
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.attn_cp_relayout.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, vp, i64p, vp, i64p, vp]
        lib.attn_cp_relayout.restype = ctypes.c_int
        lib.attn_query_status.argtypes = [vp, vp]
        lib.attn_query_status.restype = ctypes.c_int
        lib.attn_last_error.argtypes = []
        lib.attn_last_error.restype = ctypes.c_char_p
        lib.attn_last_launch_count.argtypes = []
        lib.attn_last_launch_count.restype = ctypes.c_int
        lib.attn_debug_inject.argtypes = [ctypes.c_uint, ctypes.c_int, ctypes.c_uint64]
        lib.attn_debug_inject.restype = None
        lib.attn_host_arena_size.argtypes = [P]
        lib.attn_host_arena_size.restype = sz
        lib.attn_fwd_bwd_host.argtypes = [P] + [vp] * 9 + [vp, sz, vp]
        lib.attn_fwd_bwd_host.restype = ctypes.c_int
        lib.attn_fwd_bwd_host_stages.argtypes = [P] + [vp] * 9 + [vp, sz, ctypes.c_uint, vp]
        lib.attn_fwd_bwd_host_stages.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(rc):
    if rc != 0:
        msg = load().attn_last_error().decode(errors="replace")
        raise AttnError(rc, msg)


def last_launch_count():
    return load().attn_last_launch_count()


def _code(dt):
    if dt in (torch.bfloat16, "bf16"):
        return BF16
    if dt in (torch.float16, "fp16"):
        return FP16
    if dt in (torch.float32, "fp32"):
        return FP32
    raise ValueError(f"unsupported dtype {dt}")


def _strides(t, thd):
    if t is None:
        return (0, 0, 0)
    if t.stride(-1) != 1:
        raise ValueError("the head-dim axis must be contiguous")
    if thd:
        return (0, t.stride(0), t.stride(1))
    return (t.stride(0), t.stride(1), t.stride(2))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_params(q, k, v, *, causal=True, scale=None, window=(-1, -1), bottom_right=False,
                cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None,
                o=None, dout=None, dq=None, dk=None, dv=None, o_dtype=None, grad_dtype=None,
                lse_strides=(0, 0), accumulate=False, seqused_q=None, seqused_k=None,
                bwd_ds=0):
    """attn_params_t for these tensors.  ``bwd_ds``: 0 auto, 1 always, -1
    never keep dS in the backward's workspace (attn_bwd_path)."""
    thd = cu_seqlens_q is not None
    p = Params()
    p.dtype = _code(q.dtype)
    p.o_dtype = _code(o_dtype if o_dtype is not None else (o.dtype if o is not None else q.dtype))
    p.grad_dtype = _code(grad_dtype if grad_dtype is not None else q.dtype)
    if thd:
        if cu_seqlens_k is None:
            cu_seqlens_k = cu_seqlens_q
        p.batch = cu_seqlens_q.numel() - 1
        p.cu_seqlens_q = cu_seqlens_q.data_ptr()
        p.cu_seqlens_k = cu_seqlens_k.data_ptr()
        p.total_q, p.total_k = q.shape[0], k.shape[0]
        p.seqlen_q = int(max_seqlen_q if max_seqlen_q is not None else q.shape[0])
        p.seqlen_k = int(max_seqlen_k if max_seqlen_k is not None else k.shape[0])
        hq, dqk = q.shape[1], q.shape[2]
        hkv, dvd = k.shape[1], v.shape[2]
    else:
        p.batch, p.seqlen_q, hq, dqk = q.shape
        p.seqlen_k, hkv, dvd = k.shape[1], k.shape[2], v.shape[3]
    p.heads_q, p.heads_kv, p.d_qk, p.d_v = hq, hkv, dqk, dvd
    for name, t in (("stride_q", q), ("stride_k", k), ("stride_v", v), ("stride_o", o),
                    ("stride_do", dout), ("stride_dq", dq), ("stride_dk", dk),
                    ("stride_dv", dv)):
        getattr(p, name)[:] = _strides(t, thd)
    p.stride_lse[:] = lse_strides
    p.causal = int(bool(causal))
    p.bottom_right = int(bool(bottom_right))
    p.window_left, p.window_right = int(window[0]), int(window[1])
    p.softmax_scale = float(scale if scale is not None else 1.0 / math.sqrt(dqk))
    p.accumulate = int(bool(accumulate))
    p.bwd_ds = int(bwd_ds)
    if seqused_q is not None:  # padded THD: device int32 [batch] visible lengths
        p.seqused_q = seqused_q.data_ptr()
        p.seqused_k = (seqused_k if seqused_k is not None else seqused_q).data_ptr()
    return p


def _lse_shape(q, thd):
    if thd:
        return (q.shape[1], q.shape[0])
    return (q.shape[0], q.shape[2], q.shape[1])


def fwd(q, k, v, *, causal=True, scale=None, window=(-1, -1), bottom_right=False,
        cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None,
        seqused_q=None, seqused_k=None, out=None, lse=None, o_dtype=None, lse_strides=(0, 0),
        workspace=None, stream=None):
    """Fused attention forward. Returns (o, lse).  lse_strides: element strides
    {batch, head} of `lse` ((0, 0) = its default layout)."""
    lib = load()
    thd = cu_seqlens_q is not None
    odt = o_dtype if o_dtype is not None else (out.dtype if out is not None else q.dtype)
    if out is None:
        shape = (*q.shape[:-2], q.shape[-2], v.shape[-1])
        out = torch.empty(shape, dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty(_lse_shape(q, thd), dtype=torch.float32, device=q.device)
    p = make_params(q, k, v, causal=causal, scale=scale, window=window,
                    bottom_right=bottom_right, cu_seqlens_q=cu_seqlens_q,
                    cu_seqlens_k=cu_seqlens_k, max_seqlen_q=max_seqlen_q,
                    max_seqlen_k=max_seqlen_k, o=out, o_dtype=odt, lse_strides=lse_strides,
                    seqused_q=seqused_q, seqused_k=seqused_k)
    need = lib.attn_fwd_workspace_size(ctypes.byref(p))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.attn_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def bwd(q, k, v, o, dout, lse, *, causal=True, scale=None, window=(-1, -1),
        bottom_right=False, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None,
        max_seqlen_k=None, seqused_q=None, seqused_k=None, dq=None, dk=None, dv=None,
        grad_dtype=None, lse_strides=(0, 0), accumulate=False, workspace=None, stream=None,
        stage="all", bwd_ds=0):
    """Fused attention backward. Returns (dq, dk, dv).

    ``stage``: "all" (attn_bwd), or one of "preprocess", "dq", "dkdv" to run a
    single stage of it (the C ABI's attn_bwd_* entry points; on the BWD_DS
    path the dkdv stage comes before the dq stage).  ``bwd_ds``: see
    make_params."""
    lib = load()
    gdt = grad_dtype if grad_dtype is not None else q.dtype
    if dq is None:
        dq = torch.empty(q.shape, dtype=gdt, device=q.device)
    if dk is None:
        dk = torch.empty(k.shape, dtype=gdt, device=q.device)
    if dv is None:
        dv = torch.empty(v.shape, dtype=gdt, device=q.device)
    p = make_params(q, k, v, causal=causal, scale=scale, window=window,
                    bottom_right=bottom_right, cu_seqlens_q=cu_seqlens_q,
                    cu_seqlens_k=cu_seqlens_k, max_seqlen_q=max_seqlen_q,
                    max_seqlen_k=max_seqlen_k, o=o, dout=dout, dq=dq, dk=dk, dv=dv,
                    o_dtype=o.dtype, grad_dtype=gdt, lse_strides=lse_strides,
                    accumulate=accumulate, seqused_q=seqused_q, seqused_k=seqused_k,
                    bwd_ds=bwd_ds)
    need = lib.attn_bwd_workspace_size(ctypes.byref(p))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    fn = {"all": lib.attn_bwd, "preprocess": lib.attn_bwd_preprocess, "dq": lib.attn_bwd_dq,
          "dkdv": lib.attn_bwd_dkdv}[stage]
    _check(fn(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout),
                        _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                        workspace.numel(), _stream(stream)))
    return dq, dk, dv


def bwd_noalloc(q, k, v, o, dout, lse, *, causal=True, scale=None, window=(-1, -1),
                bottom_right=False, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None,
                max_seqlen_k=None, dq=None, dk=None, dv=None, grad_dtype=None,
                lse_strides=(0, 0), accumulate=False, stream=None):
    """attn_bwd_noalloc: the backward without a caller workspace.

    For callers that must not allocate device memory while they run (the
    library's own 8 MiB static scratch area is used instead; concurrent calls
    on one device race).  The output tensors are still the caller's.
    Returns (dq, dk, dv)."""
    lib = load()
    gdt = grad_dtype if grad_dtype is not None else q.dtype
    if dq is None:
        dq = torch.empty(q.shape, dtype=gdt, device=q.device)
    if dk is None:
        dk = torch.empty(k.shape, dtype=gdt, device=q.device)
    if dv is None:
        dv = torch.empty(v.shape, dtype=gdt, device=q.device)
    p = make_params(q, k, v, causal=causal, scale=scale, window=window,
                    bottom_right=bottom_right, cu_seqlens_q=cu_seqlens_q,
                    cu_seqlens_k=cu_seqlens_k, max_seqlen_q=max_seqlen_q,
                    max_seqlen_k=max_seqlen_k, o=o, dout=dout, dq=dq, dk=dk, dv=dv,
                    o_dtype=o.dtype, grad_dtype=gdt, lse_strides=lse_strides,
                    accumulate=accumulate)
    _check(lib.attn_bwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout),
                                _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))
    return dq, dk, dv


def _host_params(q, k, v, dout, o, dq, dk, dv, kw):
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout), ("o", o), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
    return make_params(q, k, v, o=o, dout=dout, dq=dq, dk=dk, dv=dv, o_dtype=o.dtype,
                       grad_dtype=dq.dtype, **kw)


def host_arena_size(q, k, v, dout, o, dq, dk, dv, **kw):
    """Bytes of device arena attn_fwd_bwd_host needs for these host tensors."""
    p = _host_params(q, k, v, dout, o, dq, dk, dv, kw)
    return load().attn_host_arena_size(ctypes.byref(p))


def fwd_bwd_host(q, k, v, dout, o, lse, dq, dk, dv, arena, *, stream=None, stages=HOST_ALL,
                 **kw):
    """attn_fwd_bwd_host: one forward + backward step whose inputs (q, k, v,
    dout) and outputs (o, lse, dq, dk, dv) are HOST tensors (pinned for the
    copies to overlap); ``arena`` is a device uint8 tensor of at least
    host_arena_size() bytes.  THD ``cu_seqlens_q/k`` (and ``seqused_q/k``) in
    ``kw`` are host int32 tensors too.  Enqueued on ``stream``; the outputs are
    valid once it has passed the call.  ``stages``: a mask of HOST_UPLOAD,
    HOST_COMPUTE and HOST_DOWNLOAD (attn_fwd_bwd_host_stages) to run part of
    the step, e.g. to pipeline consecutive steps over several streams."""
    lib = load()
    if lse.is_cuda or not arena.is_cuda:
        raise ValueError("lse must be a host tensor and arena a device tensor")
    p = _host_params(q, k, v, dout, o, dq, dk, dv, kw)
    args = (ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(lse),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(arena), arena.numel())
    if stages == HOST_ALL:
        _check(lib.attn_fwd_bwd_host(*args, _stream(stream)))
    else:
        _check(lib.attn_fwd_bwd_host_stages(*args, int(stages), _stream(stream)))
    return o, lse, dq, dk, dv


def bwd_path(q, k, v, **kw):
    """attn_bwd_path: BWD_RECOMPUTE, BWD_DS or BWD_PDS for these tensors."""
    p = make_params(q, k, v, **kw)
    r = load().attn_bwd_path(ctypes.byref(p))
    if r < 0:
        raise AttnError(1, load().attn_last_error().decode(errors="replace"))
    return r


def workspace_size(kind, q, k, v, **kw):
    """Bytes of workspace attn_fwd ('fwd') or attn_bwd ('bwd') needs."""
    p = make_params(q, k, v, **kw)
    fn = load().attn_fwd_workspace_size if kind == "fwd" else load().attn_bwd_workspace_size
    return fn(ctypes.byref(p))


def lse_merge(o_parts, lse_parts, row0, nrows, rows, *, out=None, lse_out=None,
              out_dtype=torch.bfloat16, stream=None):
    """LSE-weighted merge.  o_parts[i]: fp32 [nrows[i], H, dv]; lse_parts[i]: fp32
    [H, nrows[i]]; part i covers output rows [row0[i], row0[i] + nrows[i])."""
    lib = load()
    n = len(o_parts)
    heads, dvd = o_parts[0].shape[1], o_parts[0].shape[2]
    if out is None:
        out = torch.empty((rows, heads, dvd), dtype=out_dtype, device=o_parts[0].device)
    if lse_out is None:
        lse_out = torch.empty((heads, rows), dtype=torch.float32, device=o_parts[0].device)
    optrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in o_parts])
    lptrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in lse_parts])
    r0 = (ctypes.c_int64 * n)(*[int(x) for x in row0])
    nr = (ctypes.c_int64 * n)(*[int(x) for x in nrows])
    _check(lib.attn_lse_merge(n, optrs, lptrs, r0, nr, int(rows), int(heads), int(dvd),
                              _ptr(out), _code(out.dtype), _ptr(lse_out), _stream(stream)))
    return out, lse_out


def debug_inject(kernel_mask, drop_load, wait_limit_ns=0):
    """TEST ONLY: arm attn_debug_inject for the next attn_fwd / attn_bwd call on
    this thread (the first CTA of each selected kernel leaves out load
    ``drop_load`` and waits at most ``wait_limit_ns``; 0 keeps 2 s)."""
    load().attn_debug_inject(int(kernel_mask), int(drop_load), int(wait_limit_ns))


def query_status(workspace, stream=None):
    """Synchronise the stream and raise if the device status word is set."""
    _check(load().attn_query_status(_ptr(workspace), _stream(stream)))


def cp_relayout(src, dst, *, to_heads, cp, stream=None):
    """All-to-all CP relayout between sequence shards and head shards.

    Token-major tensors (Q, K, V, O, dO, gradients): sequence side
    [cp, 2*chunk, heads, d], head side [cp, seqlen, heads/cp, d].
    LSE-like FP32 tensors (head-major): sequence side [cp, heads, 2*chunk],
    head side [cp, heads/cp, seqlen].  to_heads: src is the sequence side."""
    seq, head = (src, dst) if to_heads else (dst, src)
    if seq.dim() == 4:  # [cp, tokens, heads, d]
        seqlen, heads, d = head.shape[1], seq.shape[2], seq.shape[3]
        ss = (seq.stride(0), seq.stride(1), seq.stride(2))
        hs = (head.stride(0), head.stride(1), head.stride(2))
        assert seq.stride(3) == 1 and head.stride(3) == 1, "d must be contiguous"
    else:  # [cp, heads, tokens]
        seqlen, heads, d = head.shape[2], seq.shape[1], 1
        ss = (seq.stride(0), seq.stride(2), seq.stride(1))
        hs = (head.stride(0), head.stride(2), head.stride(1))
    assert src.dtype == dst.dtype
    arr = ctypes.c_int64 * 3
    s_src, s_dst = (arr(*ss), arr(*hs)) if to_heads else (arr(*hs), arr(*ss))
    _check(load().attn_cp_relayout(int(bool(to_heads)), cp, seqlen, heads, d, src.element_size(),
                                   _ptr(src), s_src, _ptr(dst), s_dst, _stream(stream)))
    return dst
