"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark uses, on outputs the oracle can compute exactly from a sub-problem:

* a block of query rows [a, b) of a causal problem sees keys [0, b) (window:
  [a - L, b)); it is exactly a bottom-right-aligned problem with those keys,
  so O, LSE and dQ of the block come out exact;
* key rows [a, S) at the end of a causal sequence only receive gradient from
  query rows >= a, so their dK/dV come out exact from the query block [a, S);
* with MHA a head is independent of the others, and with GQA a key/value head
  together with its query heads is;
* dK/dV of any key block, including the deepest accumulations (key block 0 of
  a causal sequence sums over every query tile of every head of its group),
  come out exact from the oracle's key-subset backward, which runs the full
  forward of every query row that sees a selected key.
Every sample is gated with the 2x-naive criterion against the naive
implementation run on the same sub-problem (or key subset), and gradients by
relative L2.  The GPU results come from one call at the full size, in the
launch configuration the benchmark uses.
"""

import numpy as np
import pytest
import torch

import oracle
from bwd_tcgen05_tmem_gb300 import attn, synth
from parity import check_lse, gate, rel_l2

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


_RUNS = {}


def run_dense(w):
    """One full-size forward + backward of workload `w` on the GPU (cached for
    the tests of this module; inputs and results on the CPU)."""
    if w.name in _RUNS:
        return _RUNS[w.name]
    inp = synth.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = attn.fwd(q, k, v, causal=True, scale=w.scale, window=w.window)
    g = attn.bwd(q, k, v, o, do, lse, causal=True, scale=w.scale, window=w.window)
    torch.cuda.synchronize()
    _RUNS[w.name] = (inp, o.cpu(), lse.cpu(), [t.cpu() for t in g])
    del q, k, v, do, o, lse, g
    torch.cuda.empty_cache()
    return _RUNS[w.name]


def check_key_blocks(q, k, v, do, dk, dv, key_rows, *, scale, window=(-1, -1), dtype="bf16",
                     cu=None):
    """dK/dV of `key_rows` against the oracle's key-subset backward and the
    naive floor on the same subset.  q/k/v/do: CPU tensors [T, H, d] of one
    problem (a head group, or all heads); dk/dv: the GPU's gradients, same
    layout.  `cu`: sequence offsets (None: one sequence)."""
    t = q.shape[0]
    cu = [0, t] if cu is None else cu
    qs, ks, vs, ds = (f64(x) for x in (q, k, v, do))
    kw = dict(scale=scale, causal=True, window=window, key_rows=key_rows)
    ek, ev = oracle.bwd_kv(qs, ks, vs, ds, cu, cu, **kw)
    nk, nv = oracle.naive_kv(qs, ks, vs, ds, cu, cu, dtype=dtype, **kw)
    rows = np.asarray(list(key_rows))
    for name, got, ex, nv_ in (("dk", dk, ek, nk), ("dv", dv, ev, nv)):
        g_ = f64(got)[rows]
        gate(name, g_, ex[rows], np.max(np.abs(nv_[rows] - ex[rows])))
        rel_l2(name, g_, ex[rows])


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


# ------------------------------------------------------------------ deep dK/dV
# Key block 0 of a causal sequence is the deepest accumulation of the dK/dV
# kernels (every query tile of every query head of its group); a middle block
# gets half of them.  These tests check those blocks at the full sizes.


def test_b1_h32_s32768_d192_128_deep_key_blocks():
    """Key blocks 0 and 96 (512 and 320 query tiles of 64 rows) and the last
    block, heads 0 and 31, against the oracle over all 32768 query rows."""
    w = synth.WORKLOADS["b1_h32_s32768_d192_128"]
    inp, _, _, (_, dk, dv) = run_dense(w)
    S = w.seqlen
    heads = [0, w.heads_q - 1]  # MHA: each head is its own group
    key_rows = list(range(0, 128)) + list(range(12288, 12416)) + list(range(S - 128, S))
    sl = lambda t: t[0][:, heads]  # noqa: E731
    check_key_blocks(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["dout"]), sl(dk), sl(dv),
                     key_rows, scale=w.scale)


def test_b1_h16_kv4_s16384_d512_deep_key_blocks():
    """d512 GQA: key blocks 0, 64 and the last one of kv head 3, summed over its
    four query heads and all their query tiles (the materialising dK/dV GEMMs)."""
    w = synth.WORKLOADS["b1_h16_kv4_s16384_d512"]
    inp, _, _, (_, dk, dv) = run_dense(w)
    S = w.seqlen
    grp = w.heads_q // w.heads_kv
    g = w.heads_kv - 1
    hs = slice(g * grp, (g + 1) * grp)
    key_rows = list(range(0, 128)) + list(range(8192, 8320)) + list(range(S - 128, S))
    check_key_blocks(inp["q"][0, :, hs], inp["k"][0, :, g:g + 1], inp["v"][0, :, g:g + 1],
                     inp["dout"][0, :, hs], dk[0, :, g:g + 1], dv[0, :, g:g + 1], key_rows,
                     scale=w.scale)


def test_b1_h16_kv4_s16384_d256_window1024_deep_key_blocks():
    """Windowed d256: interior key blocks, whose dK/dV sum over every query tile
    the window lets see them, for all four query heads of kv heads 0 and 3."""
    w = synth.WORKLOADS["b1_h16_kv4_s16384_d256_w1024"]
    inp, _, _, (_, dk, dv) = run_dense(w)
    grp = w.heads_q // w.heads_kv
    key_rows = list(range(0, 128)) + list(range(8064, 8192)) + list(range(12000, 12128))
    for g in (0, w.heads_kv - 1):
        hs = slice(g * grp, (g + 1) * grp)
        check_key_blocks(inp["q"][0, :, hs], inp["k"][0, :, g:g + 1], inp["v"][0, :, g:g + 1],
                         inp["dout"][0, :, hs], dk[0, :, g:g + 1], dv[0, :, g:g + 1], key_rows,
                         scale=w.scale, window=w.window)


def test_thd_h32_kv8_t65536_d128_longest_document_deep_key_blocks():
    """Packed THD: the first, a middle and the last key block of the longest
    document, kv heads 0 and 7 with their query heads."""
    w = synth.WORKLOADS["thd_h32_kv8_t65536_d128_bf16"]
    inp = synth.make_inputs(w)
    cu = inp["cu_seqlens"]
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    cud = cu.cuda()
    kw = dict(causal=True, scale=w.scale, cu_seqlens_q=cud, cu_seqlens_k=cud,
              max_seqlen_q=inp["max_seqlen"], max_seqlen_k=inp["max_seqlen"])
    o, lse = attn.fwd(q, k, v, **kw)
    _, dk, dv = attn.bwd(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    dk, dv = dk.cpu(), dv.cpu()
    lens = (cu[1:] - cu[:-1]).tolist()
    doc = max(range(len(lens)), key=lambda i: lens[i])
    a, b = int(cu[doc]), int(cu[doc + 1])
    n = b - a
    mid = (n // 2) // 128 * 128
    key_rows = list(range(0, 128)) + list(range(mid, mid + 128)) + list(range(n - 128, n))
    grp = w.heads_q // w.heads_kv
    for g in (0, w.heads_kv - 1):
        hs = slice(g * grp, (g + 1) * grp)
        check_key_blocks(inp["q"][a:b, hs], inp["k"][a:b, g:g + 1], inp["v"][a:b, g:g + 1],
                         inp["dout"][a:b, hs], dk[a:b, g:g + 1], dv[a:b, g:g + 1], key_rows,
                         scale=w.scale)
