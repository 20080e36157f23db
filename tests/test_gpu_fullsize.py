"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark uses, on outputs the oracle can compute exactly from a sub-problem:

* a block of query rows [a, b) of a causal problem sees keys [0, b) (window:
  [a - L, b)); it is exactly a bottom-right-aligned problem with those keys,
  so O, LSE and dQ of the block come out exact;
* key rows [a, S) at the end of a causal sequence only receive gradient from
  query rows >= a, so their dK/dV come out exact from the query block [a, S);
* with MHA a head is independent of the others, and with GQA a key/value head
  together with its query heads is.
Every sample is gated with the 2x-naive criterion against the naive
implementation run on the same sub-problem, and gradients by relative L2.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from bwd_tcgen05_tmem_gb300 import attn, synth
from parity import GRAD_REL_L2, check_lse, gate, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from bwd_tcgen05_tmem_gb300 import build
    build.build()
    attn.load()


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def sub_reference(q, k, v, do, rows, keys, *, scale, window=(-1, -1), dtype="bf16"):
    """Oracle + naive floor of query rows `rows` against keys `keys` (ranges of
    one sequence; q/k/v/do are [S, H, d] CPU tensors of one head group)."""
    qs, ks, vs, ds = (f64(t) for t in (q[rows], k[keys], v[keys], do[rows]))
    nq, nk = qs.shape[0], ks.shape[0]
    kw = dict(scale=scale, causal=True, window=window, bottom_right=True)
    o, lse = oracle.fwd(qs, ks, vs, [0, nq], [0, nk], **kw)
    dq, dk, dv = oracle.bwd(qs, ks, vs, ds, [0, nq], [0, nk], **kw)
    nres = oracle.naive(qs, ks, vs, [0, nq], [0, nk], dtype=dtype, dout=ds, **kw)
    floors = {"o": np.max(np.abs(nres[0] - o)), "dq": np.max(np.abs(nres[2] - dq)),
              "dk": np.max(np.abs(nres[3] - dk)), "dv": np.max(np.abs(nres[4] - dv))}
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, floor=floors, nres=nres)


def check_block(got, ref, tail_keys=None):
    gate("o", got["o"], ref["o"], ref["floor"]["o"])
    check_lse(got["lse"], ref["lse"])
    gate("dq", got["dq"], ref["dq"], ref["floor"]["dq"])
    rel_l2("dq", got["dq"], ref["dq"])
    if tail_keys is not None:  # the last rows of the key block are exact
        for name in ("dk", "dv"):
            ex = ref[name][tail_keys]
            fl = np.max(np.abs(ref["nres"][3 if name == "dk" else 4][tail_keys] - ex))
            gate(name, got[name], ex, fl)
            rel_l2(name, got[name], ex)


def run_dense(w):
    inp = synth.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = attn.fwd(q, k, v, causal=True, scale=w.scale, window=w.window)
    g = attn.bwd(q, k, v, o, do, lse, causal=True, scale=w.scale, window=w.window)
    torch.cuda.synchronize()
    return inp, o.cpu(), lse.cpu(), [t.cpu() for t in g]


def test_b2_h32_s4096_d192_128_two_full_heads():
    w = synth.WORKLOADS["b2_h32_s4096_d192_128"]
    inp, o, lse, (dq, dk, dv) = run_dense(w)
    S = w.seqlen
    heads = [0, w.heads_q - 1]  # MHA: each head is an independent problem
    for b in range(w.batch):
        sl = lambda t: t[b][:, heads]  # noqa: E731
        ref = sub_reference(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["dout"]),
                            slice(0, S), slice(0, S), scale=w.scale)
        got = dict(o=sl(o), lse=lse[b][heads], dq=sl(dq), dk=sl(dk), dv=sl(dv))
        check_block(got, ref, tail_keys=slice(0, S))


def test_b1_h32_s32768_d192_128_sampled_rows():
    w = synth.WORKLOADS["b1_h32_s32768_d192_128"]
    inp, o, lse, (dq, dk, dv) = run_dense(w)
    S, n = w.seqlen, 192
    heads = [0, w.heads_q - 1]
    sl = lambda t: t[0][:, heads]  # noqa: E731
    for a in (0, 12345, S - n):
        rows = slice(a, a + n)
        ref = sub_reference(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["dout"]),
                            rows, slice(0, a + n), scale=w.scale)
        tail = slice(a, a + n) if a == S - n else None
        got = dict(o=sl(o)[rows], lse=lse[0][heads][:, rows], dq=sl(dq)[rows],
                   dk=sl(dk)[a:a + n], dv=sl(dv)[a:a + n])
        check_block(got, ref, tail_keys=tail)


def test_b1_h16_kv4_s16384_d256_window1024_sampled_rows():
    w = synth.WORKLOADS["b1_h16_kv4_s16384_d256_w1024"]
    inp, o, lse, (dq, dk, dv) = run_dense(w)
    S, n, L = w.seqlen, 256, w.window[0]
    grp = w.heads_q // w.heads_kv
    for g in (0, w.heads_kv - 1):
        hs = slice(g * grp, (g + 1) * grp)
        for a in (100, 7000, S - n):
            lo = max(0, a - L)
            rows = slice(a, a + n)
            ref = sub_reference(inp["q"][0, :, hs], inp["k"][0, :, g:g + 1],
                                inp["v"][0, :, g:g + 1], inp["dout"][0, :, hs], rows,
                                slice(lo, a + n), scale=w.scale, window=w.window)
            tail = slice(a - lo, a - lo + n) if a == S - n else None
            got = dict(o=o[0, rows, hs], lse=lse[0, hs, rows], dq=dq[0, rows, hs],
                       dk=dk[0, a:a + n, g:g + 1], dv=dv[0, a:a + n, g:g + 1])
            check_block(got, ref, tail_keys=tail)


def test_b1_h16_kv4_s16384_d512_sampled_rows():
    w = synth.WORKLOADS["b1_h16_kv4_s16384_d512"]
    inp, o, lse, (dq, dk, dv) = run_dense(w)
    S, n = w.seqlen, 128
    grp = w.heads_q // w.heads_kv
    g = w.heads_kv - 1
    hs = slice(g * grp, (g + 1) * grp)
    for a in (0, 8000, S - n):
        rows = slice(a, a + n)
        ref = sub_reference(inp["q"][0, :, hs], inp["k"][0, :, g:g + 1], inp["v"][0, :, g:g + 1],
                            inp["dout"][0, :, hs], rows, slice(0, a + n), scale=w.scale)
        tail = slice(a, a + n) if a == S - n else None
        got = dict(o=o[0, rows, hs], lse=lse[0, hs, rows], dq=dq[0, rows, hs],
                   dk=dk[0, a:a + n, g:g + 1], dv=dv[0, a:a + n, g:g + 1])
        check_block(got, ref, tail_keys=tail)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_thd_h32_kv8_t65536_d128_sampled_documents(dtype):
    w = synth.WORKLOADS[f"thd_h32_kv8_t65536_d128_{dtype}"]
    inp = synth.make_inputs(w)
    cu = inp["cu_seqlens"]
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    cud = cu.cuda()
    kw = dict(causal=True, scale=w.scale, cu_seqlens_q=cud, cu_seqlens_k=cud,
              max_seqlen_q=inp["max_seqlen"], max_seqlen_k=inp["max_seqlen"])
    o, lse = attn.fwd(q, k, v, **kw)
    dq, dk, dv = attn.bwd(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    o, lse, dq, dk, dv = (t.cpu() for t in (o, lse, dq, dk, dv))
    lens = (cu[1:] - cu[:-1]).tolist()
    order = sorted(range(len(lens)), key=lambda i: lens[i])
    grp = w.heads_q // w.heads_kv
    for doc in (order[0], order[1]):  # the two shortest documents (one is the cut tail)
        a, b = int(cu[doc]), int(cu[doc + 1])
        for g in (0, w.heads_kv - 1):
            hs = slice(g * grp, (g + 1) * grp)
            ref = sub_reference(inp["q"][a:b, hs], inp["k"][a:b, g:g + 1], inp["v"][a:b, g:g + 1],
                                inp["dout"][a:b, hs], slice(0, b - a), slice(0, b - a),
                                scale=w.scale, dtype=dtype)
            got = dict(o=o[a:b, hs], lse=lse[hs, a:b], dq=dq[a:b, hs], dk=dk[a:b, g:g + 1],
                       dv=dv[a:b, g:g + 1])
            check_block(got, ref, tail_keys=slice(0, b - a))
