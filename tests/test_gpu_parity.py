"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Sizes span several 128-row tiles with a ragged tail; cases cover every head
dim pair, MHA and GQA, BF16 and FP16, dense and packed THD (with empty and
one-token documents), causal top-left / bottom-right, sliding windows,
non-causal attention and rows that see no key.
"""
import math

import numpy as np
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


def dense_inputs(b, sq, sk, hq, hkv, dqk, dv, dtype):
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    q = synth.normal((b, sq, hq, dqk), synth.SEED_Q, dt)
    k = synth.normal((b, sk, hkv, dqk), synth.SEED_K, dt)
    v = synth.normal((b, sk, hkv, dv), synth.SEED_V, dt)
    do = synth.normal((b, sq, hq, dv), synth.SEED_DO, dt)
    return q, k, v, do


def run_and_check(q, k, v, do, *, dtype, causal=True, window=(-1, -1), bottom_right=False,
                  cu=None, max_len=None, backward=True, bwd_ds=0, grads=False):
    scale = 1.0 / math.sqrt(q.shape[-1])
    dev = "cuda"
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    kw = dict(causal=causal, scale=scale, window=window, bottom_right=bottom_right)
    if cu is not None:
        cud = cu.to(dev)
        kw.update(cu_seqlens_q=cud, cu_seqlens_k=cud, max_seqlen_q=max_len, max_seqlen_k=max_len)
    o, lse = attn.fwd(qd, kd, vd, **kw)
    torch.cuda.synchronize()
    ref = Reference(q, k, v, do if backward else None, causal=causal, scale=scale,
                    window=window, bottom_right=bottom_right, cu_q=cu, cu_k=cu, dtype=dtype)
    report = {}
    gate("o", o, ref.o, ref.floor["o"], report)
    check_lse(lse, ref.lse)
    if backward:
        dq, dk, dv = attn.bwd(qd, kd, vd, o, dod, lse, bwd_ds=bwd_ds, **kw)
        torch.cuda.synchronize()
        for name, got, ex in (("dq", dq, ref.dq), ("dk", dk, ref.dk), ("dv", dv, ref.dv)):
            gate(name, got, ex, ref.floor[name], report)
            rel_l2(name, got, ex)
        if grads:
            report["grads"] = (dq, dk, dv)
    return report


DENSE = [
    # b, sq, sk, hq, hkv, dqk, dv, dtype, causal, window, bottom_right
    (2, 300, 300, 2, 2, 64, 64, "bf16", True, (-1, -1), False),
    (2, 300, 300, 2, 2, 128, 128, "bf16", True, (-1, -1), False),
    (2, 300, 300, 2, 2, 192, 128, "bf16", True, (-1, -1), False),
    (1, 300, 300, 2, 2, 256, 256, "bf16", True, (-1, -1), False),
    (2, 300, 300, 8, 2, 128, 128, "fp16", True, (-1, -1), False),
    (1, 300, 300, 6, 2, 192, 128, "fp16", True, (-1, -1), False),
    (1, 400, 400, 4, 1, 256, 256, "bf16", True, (100, 0), False),
    (1, 200, 333, 2, 2, 128, 128, "bf16", True, (-1, -1), True),
    (1, 333, 200, 2, 2, 128, 128, "bf16", True, (-1, -1), True),
    (1, 300, 300, 2, 2, 128, 128, "bf16", False, (-1, -1), False),
    (1, 300, 300, 2, 2, 64, 64, "bf16", False, (30, 20), False),
    (1, 130, 130, 2, 2, 64, 64, "bf16", True, (0, 0), False),
    # head dim 512: the materialising backward
    (1, 260, 260, 4, 1, 512, 512, "bf16", True, (-1, -1), False),
    (2, 200, 333, 2, 2, 512, 512, "fp16", True, (-1, -1), True),
    (1, 300, 300, 2, 1, 512, 512, "bf16", False, (100, 30), False),
]


@pytest.mark.parametrize("case", DENSE, ids=lambda c: f"b{c[0]}q{c[1]}k{c[2]}h{c[3]}/{c[4]}d{c[5]}-{c[6]}{c[7]}c{int(c[8])}w{c[9][0]}br{int(c[10])}")
def test_dense(case):
    b, sq, sk, hq, hkv, dqk, dv, dtype, causal, window, br = case
    q, k, v, do = dense_inputs(b, sq, sk, hq, hkv, dqk, dv, dtype)
    run_and_check(q, k, v, do, dtype=dtype, causal=causal, window=window, bottom_right=br)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("dims", [(128, 128), (192, 128), (64, 64), (256, 256), (512, 512)])
def test_thd_varlen(dtype, dims):
    lens = [0, 1, 129, 300, 64, 200, 0]
    w = synth.Workload("t", 0, 0, 8, 2, dims[0], dims[1], dtype=dtype, thd_total=1)
    inp = synth.make_inputs(w, lengths=lens)
    run_and_check(inp["q"], inp["k"], inp["v"], inp["dout"], dtype=dtype,
                  cu=inp["cu_seqlens"], max_len=inp["max_seqlen"])


@pytest.mark.parametrize("dims", [(128, 128), (192, 128), (512, 512)])
def test_thd_padded_seqused(dims):
    """Padded THD (TransformerEngine PR #3149: physical padded offsets plus
    visible lengths): gap rows are neither read nor written, and the visible
    rows equal the oracle run on the compacted documents."""
    used = [0, 1, 129, 300, 64, 200, 0]
    gaps = [5, 0, 7, 128, 3, 1, 9]
    padded = [u + g for u, g in zip(used, gaps)]
    cu = torch.tensor([0] + list(np.cumsum(padded)), dtype=torch.int32)
    total, hq, hkv = int(cu[-1]), 8, 2
    g = torch.Generator().manual_seed(11)
    q = torch.randn(total, hq, dims[0], generator=g).bfloat16()
    k = torch.randn(total, hkv, dims[0], generator=g).bfloat16()
    v = torch.randn(total, hkv, dims[1], generator=g).bfloat16()
    do = torch.randn(total, hq, dims[1], generator=g).bfloat16()
    su = torch.tensor(used, dtype=torch.int32)
    dev = "cuda"
    kw = dict(causal=True, cu_seqlens_q=cu.to(dev), cu_seqlens_k=cu.to(dev),
              max_seqlen_q=max(padded), max_seqlen_k=max(padded), seqused_q=su.to(dev),
              seqused_k=su.to(dev))
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    nan = float("nan")
    o = torch.full((total, hq, dims[1]), nan, dtype=torch.bfloat16, device=dev)
    lse = torch.full((hq, total), nan, device=dev)
    attn.fwd(qd, kd, vd, out=o, lse=lse, **kw)
    dq, dk, dv = (torch.full_like(t, nan) for t in (qd, kd, vd))
    attn.bwd(qd, kd, vd, o, dod, lse, dq=dq, dk=dk, dv=dv, **kw)
    torch.cuda.synchronize()
    rows = torch.cat([torch.arange(int(cu[b]), int(cu[b]) + used[b]) for b in range(len(used))])
    gap = torch.ones(total, dtype=torch.bool)
    gap[rows] = False
    for t in (o, dq, dk, dv):  # gap rows untouched
        assert torch.isnan(t.cpu()[gap].float()).all()
    assert torch.isnan(lse.cpu()[:, gap]).all()
    cu_c = [0] + list(np.cumsum(used))
    ref = Reference(q[rows], k[rows], v[rows], do[rows], causal=True,
                    scale=1.0 / math.sqrt(dims[0]), cu_q=cu_c, cu_k=cu_c, dtype="bf16")
    gate("o", o.cpu()[rows], ref.o, ref.floor["o"])
    check_lse(lse.cpu()[:, rows], ref.lse)
    for name, got, ex in (("dq", dq, ref.dq), ("dk", dk, ref.dk), ("dv", dv, ref.dv)):
        gate(name, got.cpu()[rows], ex, ref.floor[name])
        rel_l2(name, got.cpu()[rows], ex)


@pytest.mark.parametrize("dims", [(192, 128), (256, 256), (512, 512)])
def test_sbhd_strides_equal_bshd(dims):
    """Tensors are addressed through their actual strides (TransformerEngine
    PR #3527: graphs built from each tensor's actual strides, so sbhd is
    served without a transpose): SBHD-laid-out inputs, outputs and gradients
    give bit-identical results to contiguous BSHD."""
    b, s, hq, hkv = 2, 300, 4, 2
    q, k, v, do = dense_inputs(b, s, s, hq, hkv, dims[0], dims[1], "bf16")
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = attn.fwd(qd, kd, vd)
    g = attn.bwd(qd, kd, vd, o, dod, lse)
    sb = lambda t: t.permute(1, 0, 2, 3).contiguous().permute(1, 0, 2, 3)  # noqa: E731
    qs, ks, vs, dos = (sb(t) for t in (qd, kd, vd, dod))
    assert qs.stride(1) == b * hq * dims[0]  # token-major in memory
    o_s = sb(torch.empty_like(o))
    lse_s = torch.empty_like(lse)
    attn.fwd(qs, ks, vs, out=o_s, lse=lse_s)
    gs = [sb(torch.empty_like(t)) for t in (qd, kd, vd)]
    attn.bwd(qs, ks, vs, o_s, dos, lse_s, dq=gs[0], dk=gs[1], dv=gs[2])
    torch.cuda.synchronize()
    assert torch.equal(o_s, o) and torch.equal(lse_s, lse)
    for a_, b_ in zip(gs, g):
        assert torch.equal(a_, b_)


@pytest.mark.parametrize("dims", [(192, 128), (512, 512)])
def test_cuda_graph_replay_matches_eager(dims):
    """attn_fwd + attn_bwd captured in a CUDA graph: replays on new input values,
    with the outputs poisoned before each replay, equal eager calls bit for bit
    (pointers, stream and workspace are bound per call, nothing else is kept)."""
    b, s, hq, hkv = 1, 384, 4, 2
    q, k, v, do = (t.cuda() for t in dense_inputs(b, s, s, hq, hkv, dims[0], dims[1], "bf16"))
    o, lse = torch.empty(b, s, hq, dims[1], dtype=q.dtype, device="cuda"), \
        torch.empty(b, hq, s, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fws = torch.empty(attn.workspace_size("fwd", q, k, v), dtype=torch.uint8, device="cuda")
    bws = torch.empty(attn.workspace_size("bwd", q, k, v), dtype=torch.uint8, device="cuda")

    def step():
        attn.fwd(q, k, v, out=o, lse=lse, workspace=fws)
        attn.bwd(q, k, v, o, do, lse, dq=dq, dk=dk, dv=dv, workspace=bws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    g = torch.Generator(device="cuda").manual_seed(5)
    for _ in range(2):
        for t in (q, k, v, do):
            t.copy_(torch.randn(t.shape, generator=g, device="cuda").to(t.dtype))
        for t in (o, dq, dk, dv):
            t.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        step()  # eager on the same inputs
        torch.cuda.synchronize()
        for a_, b_ in zip(got, (o, lse, dq, dk, dv)):
            assert torch.equal(a_, b_)


def test_forward_bitwise_reproducible_and_stream_bound():
    q, k, v, _ = dense_inputs(1, 700, 700, 4, 4, 192, 128, "bf16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = attn.fwd(qd, kd, vd)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        outs = [attn.fwd(qd, kd, vd) for _ in range(5)]
    torch.cuda.synchronize()
    for o2, l2 in outs:
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [128, 256, 512])
def test_backward_bitwise_reproducible(d):
    q, k, v, do = dense_inputs(1, 500, 500, 4, 2, d, d, "bf16")
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.fwd(qd, kd, vd)
    g1 = attn.bwd(qd, kd, vd, o, dod, lse)
    g2 = attn.bwd(qd, kd, vd, o, dod, lse)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_causal_row0_is_v0_exactly():
    q, k, v, _ = dense_inputs(2, 257, 257, 4, 4, 128, 128, "bf16")
    o, lse = attn.fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.equal(o[:, 0].cpu(), v[:, 0])
    ref = (q[:, 0].double() * k[:, 0].double()).sum(-1) / math.sqrt(128)
    assert torch.allclose(lse[:, :, 0].cpu().double(), ref, atol=1e-4, rtol=0)


def test_outputs_fully_overwritten():
    q, k, v, do = dense_inputs(1, 300, 300, 2, 2, 128, 128, "bf16")
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o = torch.full((1, 300, 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 2, 300), float("nan"), device="cuda")
    attn.fwd(qd, kd, vd, out=o, lse=lse)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    attn.bwd(qd, kd, vd, o, dod, lse, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()


def test_keyless_rows_exact_zero():
    q, k, v, do = dense_inputs(1, 300, 100, 2, 2, 128, 128, "bf16")
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.fwd(qd, kd, vd, bottom_right=True)
    dq, dk, dv = attn.bwd(qd, kd, vd, o, dod, lse, bottom_right=True)
    torch.cuda.synchronize()
    assert torch.all(o[:, :200] == 0)
    assert torch.all(torch.isneginf(lse[:, :, :200]))
    assert torch.all(dq[:, :200] == 0)


def test_fp32_partial_output_matches():
    q, k, v, _ = dense_inputs(1, 300, 300, 2, 2, 192, 128, "bf16")
    o16, l16 = attn.fwd(q.cuda(), k.cuda(), v.cuda())
    o32, l32 = attn.fwd(q.cuda(), k.cuda(), v.cuda(), o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(l16, l32)
    assert torch.equal(o32.to(torch.bfloat16), o16)


def test_bad_cu_seqlens_reports_status():
    q = torch.zeros(64, 2, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 10, 5, 64], dtype=torch.int32, device="cuda")  # not monotone
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    o = torch.empty(64, 2, 128, dtype=torch.bfloat16, device="cuda")
    attn.fwd(q, q, q, cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=64, max_seqlen_k=64,
             out=o, workspace=ws)
    with pytest.raises(attn.AttnError) as e:
        attn.query_status(ws)
    assert e.value.code == 5


@pytest.mark.parametrize("cp,s,dims", [(8, 640, (192, 128)), (2, 520, (128, 128)),
                                       (4, 1024, (64, 64)), (2, 520, (512, 512)),
                                       (2, 512, (256, 256))])
def test_cp_ring_emulation_matches_full_attention(cp, s, dims):
    """Dual-chunk-swap ring: FP32 partials + LSE merge + per-step backward."""
    from bwd_tcgen05_tmem_gb300 import cp as cpmod
    q, k, v, do = dense_inputs(1, s, s, 4, 4, dims[0], dims[1], "bf16")
    ring = cpmod.CPRing(q.cuda(), k.cuda(), v.cuda(), do.cuda(), cp=cp)
    o_sh, lse_sh = ring.forward()
    dq_sh, dk_sh, dv_sh = ring.backward()
    torch.cuda.synchronize()
    o = cpmod.unshard(o_sh, cp).cpu()
    lse = cpmod.unshard_lse(lse_sh, cp).cpu()
    scale = 1.0 / math.sqrt(dims[0])
    ref = Reference(q, k, v, do, causal=True, scale=scale, dtype="bf16")
    gate("o", o, ref.o, ref.floor["o"])
    check_lse(lse, ref.lse)
    for name, sh, ex in (("dq", dq_sh, ref.dq), ("dk", dk_sh, ref.dk), ("dv", dv_sh, ref.dv)):
        got = cpmod.unshard(sh, cp).cpu()
        gate(name, got, ex, ref.floor[name])
        rel_l2(name, got, ex)


@pytest.mark.parametrize("cp,s,dims,wl", [(4, 1024, (192, 128), -1), (2, 520, (128, 128), -1),
                                          (4, 768, (256, 256), 200), (2, 512, (512, 512), -1),
                                          (8, 1024, (64, 64), 100)])
def test_cp_allgather_emulation_matches_full_attention(cp, s, dims, wl):
    """All-gather CP: trimmed KV, bottom-right causal (+ window), no LSE merge."""
    from bwd_tcgen05_tmem_gb300 import cp as cpmod
    q, k, v, do = dense_inputs(1, s, s, 4, 2, dims[0], dims[1], "bf16")
    ag = cpmod.CPAllGather(q.cuda(), k.cuda(), v.cuda(), do.cuda(), cp=cp, window=(wl, 0))
    o_sh, lse_sh = ag.forward()
    dq_sh, dk, dv = ag.backward()
    torch.cuda.synchronize()
    o = cpmod.unshard(o_sh, cp).cpu()
    lse = cpmod.unshard_lse(lse_sh, cp).cpu()
    scale = 1.0 / math.sqrt(dims[0])
    ref = Reference(q, k, v, do, causal=True, scale=scale, window=(wl, 0), dtype="bf16")
    gate("o", o, ref.o, ref.floor["o"])
    check_lse(lse, ref.lse)
    for name, got, ex in (("dq", cpmod.unshard(dq_sh, cp).cpu(), ref.dq), ("dk", dk.cpu(), ref.dk),
                          ("dv", dv.cpu(), ref.dv)):
        gate(name, got, ex, ref.floor[name])
        rel_l2(name, got, ex)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_cp_relayout_bit_exact(dtype):
    """Sequence shards <-> head shards: a bit-preserving permutation, checked
    against the same permutation written with torch indexing."""
    from bwd_tcgen05_tmem_gb300 import cp as cpmod
    cp, s, h, d = 4, 256, 8, 24
    g = torch.Generator().manual_seed(7)
    x = torch.randn(1, s, h, d, generator=g).to(dtype).cuda()
    seq = torch.stack([t[0] for t in cpmod.shard(x, cp)])
    heads = torch.empty(cp, s, h // cp, d, dtype=dtype, device="cuda")
    attn.cp_relayout(seq, heads, to_heads=True, cp=cp)
    ref = x[0].reshape(s, cp, h // cp, d).permute(1, 0, 2, 3)
    back = torch.empty_like(seq)
    attn.cp_relayout(heads, back, to_heads=False, cp=cp)
    # head-major FP32 rows of one element (the LSE layout)
    lse = torch.randn(1, h, s, generator=g).cuda()
    lse_seq = torch.stack([cpmod.shard(lse.transpose(1, 2), cp)[r][0].transpose(0, 1)
                           for r in range(cp)]).contiguous()
    lse_h = torch.empty(cp, h // cp, s, device="cuda")
    attn.cp_relayout(lse_seq, lse_h, to_heads=True, cp=cp)
    torch.cuda.synchronize()
    assert torch.equal(heads.view(torch.uint8), ref.contiguous().view(torch.uint8))
    assert torch.equal(back.view(torch.uint8), seq.view(torch.uint8))
    assert torch.equal(lse_h, lse[0].reshape(cp, h // cp, s))


@pytest.mark.parametrize("cp,s,dims,hkv,wl", [(4, 1024, (192, 128), 4, -1), (2, 520, (128, 128), 2, 100),
                                              (2, 512, (512, 512), 2, -1)])
def test_cp_a2a_emulation_matches_full_attention(cp, s, dims, hkv, wl):
    """All-to-all CP: relayout to head shards, full-sequence attention per rank."""
    from bwd_tcgen05_tmem_gb300 import cp as cpmod
    q, k, v, do = dense_inputs(1, s, s, 8, hkv, dims[0], dims[1], "bf16")
    a2a = cpmod.CPA2A(q.cuda(), k.cuda(), v.cuda(), do.cuda(), cp=cp, window=(wl, 0))
    o_sh, lse_sh = a2a.forward()
    g_sh = a2a.backward()
    torch.cuda.synchronize()
    un = lambda t: cpmod.unshard([x[None] for x in t], cp).cpu()  # noqa: E731
    o = un(o_sh)
    lse = cpmod.unshard_lse([x[None] for x in lse_sh], cp).cpu()
    ref = Reference(q, k, v, do, causal=True, scale=1.0 / math.sqrt(dims[0]), window=(wl, 0),
                    dtype="bf16")
    gate("o", o, ref.o, ref.floor["o"])
    check_lse(lse, ref.lse)
    for name, got, ex in zip(("dq", "dk", "dv"), g_sh, (ref.dq, ref.dk, ref.dv)):
        gate(name, un(got), ex, ref.floor[name])
        rel_l2(name, un(got), ex)


def test_cp_ring_equals_direct_path():
    """The ring emulation and the direct kernels agree closely (plumbing check)."""
    from bwd_tcgen05_tmem_gb300 import cp as cpmod
    q, k, v, do = dense_inputs(1, 2048, 2048, 4, 4, 192, 128, "bf16")
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.fwd(qd, kd, vd)
    dq, dk, dv = attn.bwd(qd, kd, vd, o, dod, lse, grad_dtype=torch.float32)
    ring = cpmod.CPRing(qd, kd, vd, dod, cp=8)
    o_sh, lse_sh = ring.forward()
    g_sh = ring.backward()
    torch.cuda.synchronize()
    assert (cpmod.unshard(o_sh, 8).float() - o.float()).abs().max().item() < 2e-2
    assert (cpmod.unshard_lse(lse_sh, 8) - lse).abs().max().item() < 1e-4
    for got, ref in zip(g_sh, (dq, dk, dv)):
        err = (cpmod.unshard(got, 8) - ref).norm() / ref.norm()
        assert err.item() < 1e-2


@pytest.mark.parametrize("dims", [(192, 128), (256, 256), (512, 512)])
def test_backward_stages_equal_full_call(dims):
    q, k, v, do = dense_inputs(1, 300, 300, 4, 2, dims[0], dims[1], "bf16")
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.fwd(qd, kd, vd)
    g1 = attn.bwd(qd, kd, vd, o, dod, lse)
    # poisoned, so that no stage can pass on what an earlier call left behind
    ws = torch.full((attn.workspace_size("bwd", qd, kd, vd),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    dq, dk, dv = (torch.empty_like(t) for t in (qd, kd, vd))
    # on the dS path the dkdv stage writes the blocks that the dq stage reads
    order = ("dkdv", "dq") if attn.bwd_path(qd, kd, vd) == attn.BWD_DS else ("dq", "dkdv")
    for stage in ("preprocess", *order):
        attn.bwd(qd, kd, vd, o, dod, lse, dq=dq, dk=dk, dv=dv, workspace=ws, stage=stage)
    torch.cuda.synchronize()
    for a, b in zip(g1, (dq, dk, dv)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("d", [128, 256, 512])
def test_fp32_gradient_accumulate(d):
    q, k, v, do = dense_inputs(1, 300, 300, 2, 2, d, d, "bf16")
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.fwd(qd, kd, vd)
    g = attn.bwd(qd, kd, vd, o, dod, lse, grad_dtype=torch.float32)
    acc = [t.clone() for t in g]
    attn.bwd(qd, kd, vd, o, dod, lse, dq=acc[0], dk=acc[1], dv=acc[2],
             grad_dtype=torch.float32, accumulate=True)
    torch.cuda.synchronize()
    for a, b in zip(acc, g):
        assert torch.equal(a, 2 * b)
