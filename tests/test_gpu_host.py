"""attn_fwd_bwd_host: one forward + backward step from host buffers.

The entry point copies host inputs into a device arena, runs attn_fwd and
attn_bwd there and copies the results back (include/attn.h).  It adds no
arithmetic, so its outputs must equal, bit for bit, those of attn_fwd +
attn_bwd on device copies of the same inputs; one case is also gated against
the FP64 oracle so that the test stands on its own.  Cases: dense GQA with a
ragged tail, packed THD (host cu_seqlens), FP32 gradient accumulation into
the caller's host values, pageable (unpinned) host memory, two steps on two
streams with two arenas, and refusal of device pointers.
"""
import ctypes
import math

import pytest
import torch

from bwd_tcgen05_tmem_gb300 import attn, synth
from parity import Reference, check_lse, gate, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from bwd_tcgen05_tmem_gb300 import build
    build.build()
    attn.load()


def inputs(shape_q, shape_kv, dv, dtype, pin=True):
    q = synth.normal(shape_q, synth.SEED_Q, dtype)
    k = synth.normal(shape_kv, synth.SEED_K, dtype)
    v = synth.normal((*shape_kv[:-1], dv), synth.SEED_V, dtype)
    do = synth.normal((*shape_q[:-1], dv), synth.SEED_DO, dtype)
    if pin:
        q, k, v, do = (t.pin_memory() for t in (q, k, v, do))
    return q, k, v, do


def host_outputs(q, k, v, grad_dtype, pin=True, lse_shape=None):
    mk = (lambda s, dt: torch.empty(s, dtype=dt, pin_memory=pin))
    o = mk((*q.shape[:-1], v.shape[-1]), q.dtype)
    lse = mk(lse_shape, torch.float32)
    return o, lse, mk(q.shape, grad_dtype), mk(k.shape, grad_dtype), mk(v.shape, grad_dtype)


def run_host(q, k, v, do, outs, stream=None, **kw):
    o, lse, dq, dk, dv = outs
    need = attn.host_arena_size(q, k, v, do, o, dq, dk, dv, **kw)
    arena = torch.empty(need, dtype=torch.uint8, device="cuda")
    attn.fwd_bwd_host(q, k, v, do, o, lse, dq, dk, dv, arena, stream=stream, **kw)
    torch.cuda.synchronize()
    attn.query_status(arena)        # the forward's status word
    attn.query_status(arena[256:])  # the backward's
    return arena


def run_device(q, k, v, do, grad_dtype, dkw, **kw):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = attn.fwd(qd, kd, vd, **dkw, **kw)
    dq, dk, dv = attn.bwd(qd, kd, vd, o, dod, lse, grad_dtype=grad_dtype, **dkw, **kw)
    torch.cuda.synchronize()
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


def assert_same(host, dev):
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), host, dev):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("dims,dtype,grad", [((192, 128), torch.bfloat16, torch.bfloat16),
                                             ((128, 128), torch.float16, torch.float32),
                                             ((512, 512), torch.bfloat16, torch.bfloat16)])
def test_dense_host_step_equals_device_path(dims, dtype, grad):
    dqk, dv = dims
    b, s, hq, hkv = 2, 300, 4, 2
    q, k, v, do = inputs((b, s, hq, dqk), (b, s, hkv, dqk), dv, dtype)
    outs = host_outputs(q, k, v, grad, lse_shape=(b, hq, s))
    run_host(q, k, v, do, outs, causal=True)
    assert_same(outs, run_device(q, k, v, do, grad, {}, causal=True))
    if dims == (192, 128):  # the same step against the FP64 oracle
        scale = 1.0 / math.sqrt(dqk)
        ref = Reference(q, k, v, do, causal=True, scale=scale,
                        dtype="bf16" if dtype == torch.bfloat16 else "fp16")
        gate("o", outs[0], ref.o, ref.floor["o"])
        check_lse(outs[1], ref.lse)
        for name, got, ex in zip(("dq", "dk", "dv"), outs[2:], (ref.dq, ref.dk, ref.dv)):
            gate(name, got, ex, ref.floor[name])
            rel_l2(name, got, ex)


def test_thd_host_step_with_host_cu_seqlens():
    lens = [300, 17, 129, 256]
    cu = synth.cu_from_lengths(lens)
    t, hq, hkv = sum(lens), 4, 1
    q, k, v, do = inputs((t, hq, 128), (t, hkv, 128), 128, torch.float16)
    outs = host_outputs(q, k, v, torch.float16, lse_shape=(hq, t))
    kw = dict(causal=True, max_seqlen_q=max(lens), max_seqlen_k=max(lens))
    run_host(q, k, v, do, outs, cu_seqlens_q=cu, cu_seqlens_k=cu, **kw)
    cud = cu.cuda()
    dev = run_device(q, k, v, do, torch.float16, dict(cu_seqlens_q=cud, cu_seqlens_k=cud), **kw)
    assert_same(outs, dev)


def test_accumulate_adds_into_host_gradients():
    b, s, hq, hkv = 1, 260, 2, 2
    q, k, v, do = inputs((b, s, hq, 192), (b, s, hkv, 192), 128, torch.bfloat16)
    outs = host_outputs(q, k, v, torch.float32, lse_shape=(b, hq, s))
    g = torch.Generator().manual_seed(9)
    prev = [torch.randn(t.shape, generator=g) for t in outs[2:]]
    for t, p in zip(outs[2:], prev):
        t.copy_(p)
    run_host(q, k, v, do, outs, causal=True, accumulate=True)
    # device path: the same accumulation into device copies of the same values
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = attn.fwd(qd, kd, vd, causal=True)
    dq, dk, dv = (p.cuda() for p in prev)
    attn.bwd(qd, kd, vd, o, dod, lse, dq=dq, dk=dk, dv=dv, grad_dtype=torch.float32,
             accumulate=True, causal=True)
    torch.cuda.synchronize()
    assert_same(outs, [t.cpu() for t in (o, lse, dq, dk, dv)])
    assert not torch.equal(outs[2], prev[0])


def test_pageable_host_memory_and_two_streams():
    """Unpinned buffers work (the copies are then synchronous); two steps on
    two streams with two arenas give the same results as one."""
    b, s, hq, hkv = 1, 384, 2, 2
    q, k, v, do = inputs((b, s, hq, 128), (b, s, hkv, 128), 128, torch.bfloat16, pin=False)
    outs_a = host_outputs(q, k, v, torch.bfloat16, pin=False, lse_shape=(b, hq, s))
    run_host(q, k, v, do, outs_a, causal=True)
    qp, kp, vp, dop = (t.pin_memory() for t in (q, k, v, do))
    outs = [host_outputs(q, k, v, torch.bfloat16, lse_shape=(b, hq, s)) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    arenas = []
    for o_, st in zip(outs, streams):
        need = attn.host_arena_size(qp, kp, vp, dop, o_[0], *o_[2:], causal=True)
        arenas.append(torch.empty(need, dtype=torch.uint8, device="cuda"))
        attn.fwd_bwd_host(qp, kp, vp, dop, *o_, arenas[-1], stream=st, causal=True)
    torch.cuda.synchronize()
    for o_ in outs:
        assert_same(o_, outs_a)


def test_device_pointer_refused():
    b, s = 1, 128
    q, k, v, do = inputs((b, s, 2, 64), (b, s, 2, 64), 64, torch.bfloat16)
    outs = host_outputs(q, k, v, torch.bfloat16, lse_shape=(b, 2, s))
    need = attn.host_arena_size(q, k, v, do, outs[0], *outs[2:], causal=True)
    arena = torch.empty(need, dtype=torch.uint8, device="cuda")
    p = attn.make_params(q, k, v, o=outs[0], dout=do, dq=outs[2], dk=outs[3], dv=outs[4],
                         causal=True)
    qd = q.cuda()
    ptrs = [qd, k, v, do, *outs]
    lib = attn.load()
    rc = lib.attn_fwd_bwd_host(ctypes.byref(p), *[ctypes.c_void_p(t.data_ptr()) for t in ptrs],
                               ctypes.c_void_p(arena.data_ptr()), need, None)
    assert rc == 1
    assert b"device memory" in lib.attn_last_error()


def test_staged_pipeline_equals_one_call():
    """attn_fwd_bwd_host_stages: upload, compute and download of consecutive
    steps on three streams, ordered by events over two arenas (the pipeline
    the benchmark's end-to-end leg runs), give the one-call results."""
    b, s, hq, hkv = 1, 300, 4, 2
    q, k, v, do = inputs((b, s, hq, 192), (b, s, hkv, 192), 128, torch.bfloat16)
    ref = host_outputs(q, k, v, torch.bfloat16, lse_shape=(b, hq, s))
    run_host(q, k, v, do, ref, causal=True)
    outs = [host_outputs(q, k, v, torch.bfloat16, lse_shape=(b, hq, s)) for _ in range(2)]
    need = attn.host_arena_size(q, k, v, do, ref[0], *ref[2:], causal=True)
    arenas = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in range(2)]
    up, comp, down = (torch.cuda.Stream() for _ in range(3))
    n = 4
    ev = [[torch.cuda.Event() for _ in range(3)] for _ in range(n)]
    for i in range(n):
        a = i % 2
        args = (q, k, v, do, *outs[a], arenas[a])
        if i >= 2:
            up.wait_event(ev[i - 2][1])
        attn.fwd_bwd_host(*args, stream=up, stages=attn.HOST_UPLOAD, causal=True)
        ev[i][0].record(up)
        comp.wait_event(ev[i][0])
        if i >= 2:
            comp.wait_event(ev[i - 2][2])
        attn.fwd_bwd_host(*args, stream=comp, stages=attn.HOST_COMPUTE, causal=True)
        ev[i][1].record(comp)
        down.wait_event(ev[i][1])
        attn.fwd_bwd_host(*args, stream=down, stages=attn.HOST_DOWNLOAD, causal=True)
        ev[i][2].record(down)
    torch.cuda.synchronize()
    for o_ in outs:
        assert_same(o_, ref)
