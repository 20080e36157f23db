"""Pins for the FP64 oracle against things other than itself (CPU only).

The oracle (``oracle/``) is the definition of fused causal attention written out
in plain C.  These tests tie it to independent facts:

* library routines: torch's float64 ``scaled_dot_product_attention``, its
  autograd, and ``torch.logsumexp`` (TransformerEngine PR #3527 review notes:
  the reference must be float64, not float32);
* central finite differences of L = sum(dO * O) for the backward;
* closed forms (Q = 0 gives uniform attention; causal row 0 returns V[0]);
* invariants (key shift, GQA = repeated MHA, THD = per-document runs, dK sums
  to zero, LSE-merge of chunked partials = full attention, window limits);
* the accuracy criterion err(kernel, fp64) <= 2 * err(naive_bf16, fp64)
  (PR #3527 description), including its mutation test: a 1 % softmax-scale
  error must be rejected.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand(*shape):
    return rng.standard_normal(shape)


def dense(x):
    """[B, S, H, d] -> THD [B*S, H, d]."""
    return x.reshape(-1, x.shape[2], x.shape[3])


def torch_ref(q, k, v, *, scale, causal, window=(-1, -1), bottom_right=False, dout=None):
    """float64 torch reference for one sequence: q [Lq,Hq,d], k/v [Lk,Hkv,d].

    Uses torch's attention with an explicit mask built from tril/triu.  Returns
    o, lse (and dq, dk, dv when dout is given)."""
    lq, hq, _ = q.shape
    lk, hkv, _ = k.shape
    grp = hq // hkv
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kt = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    vt = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    off = (lk - lq) if bottom_right else 0
    keep = torch.ones(lq, lk, dtype=torch.bool)
    if causal:
        keep &= torch.ones(lq, lk, dtype=torch.bool).tril(diagonal=off)
    if window[0] >= 0:
        keep &= torch.ones(lq, lk, dtype=torch.bool).triu(diagonal=off - window[0])
    if window[1] >= 0:
        keep &= torch.ones(lq, lk, dtype=torch.bool).tril(diagonal=off + window[1])
    kr = kt.repeat_interleave(grp, dim=1)
    vr = vt.repeat_interleave(grp, dim=1)
    qh, kh, vh = qt.transpose(0, 1), kr.transpose(0, 1), vr.transpose(0, 1)
    scores = torch.matmul(qh, kh.transpose(-1, -2)) * scale
    scores = scores.masked_fill(~keep, float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)
    o = torch.nn.functional.scaled_dot_product_attention(
        qh, kh, vh, attn_mask=keep, scale=scale)
    has = keep.any(dim=-1)
    o = torch.where(has[None, :, None], o, torch.zeros_like(o)).transpose(0, 1)
    if dout is None:
        return o.detach().numpy(), lse.detach().numpy()
    o.backward(torch.tensor(dout, dtype=torch.float64))
    return (o.detach().numpy(), lse.detach().numpy(), qt.grad.numpy(), kt.grad.numpy(),
            vt.grad.numpy())


CASES = [
    # (Lq, Lk, hq, hkv, dqk, dv, causal, window, bottom_right)
    (17, 17, 2, 2, 8, 8, True, (-1, -1), False),
    (17, 17, 4, 2, 8, 4, True, (-1, -1), False),
    (13, 13, 2, 1, 6, 6, False, (-1, -1), False),
    (19, 19, 2, 2, 8, 8, True, (4, 0), False),
    (19, 19, 2, 2, 8, 8, False, (3, 2), False),
    (7, 15, 2, 2, 8, 8, True, (-1, -1), True),
    (15, 7, 2, 2, 8, 8, True, (-1, -1), True),
    (9, 14, 3, 1, 8, 8, True, (2, 0), True),
]


@pytest.mark.parametrize("case", CASES)
def test_matches_torch_float64(case):
    lq, lk, hq, hkv, dqk, dv, causal, window, br = case
    q, k, v = rand(lq, hq, dqk), rand(lk, hkv, dqk), rand(lk, hkv, dv)
    do = rand(lq, hq, dv)
    scale = 1.0 / math.sqrt(dqk)
    o_t, lse_t, dq_t, dk_t, dv_t = torch_ref(q, k, v, scale=scale, causal=causal,
                                            window=window, bottom_right=br, dout=do)
    kw = dict(scale=scale, causal=causal, window=window, bottom_right=br)
    o, lse = oracle.fwd(q, k, v, [0, lq], [0, lk], **kw)
    np.testing.assert_allclose(o, o_t, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lse_t))
    fin = np.isfinite(lse_t)
    np.testing.assert_allclose(lse[fin], lse_t[fin], rtol=0, atol=1e-12)
    dq, dk, dvv = oracle.bwd(q, k, v, do, [0, lq], [0, lk], **kw)
    np.testing.assert_allclose(dq, dq_t, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, dk_t, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dvv, dv_t, rtol=0, atol=1e-11)


def test_causal_top_left_matches_library_is_causal():
    """torch's own is_causal flag (top-left) with no hand-built mask."""
    q, k, v = rand(23, 2, 8), rand(23, 2, 8), rand(23, 2, 8)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q).transpose(0, 1), torch.tensor(k).transpose(0, 1),
        torch.tensor(v).transpose(0, 1), is_causal=True, scale=0.3).transpose(0, 1)
    o, _ = oracle.fwd(q, k, v, [0, 23], [0, 23], scale=0.3, causal=True)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def _loss(q, k, v, do, cu_q, cu_k, **kw):
    o, _ = oracle.fwd(q, k, v, cu_q, cu_k, **kw)
    return float(np.sum(o * do))


FD_CASES = [
    ([0, 6], [0, 6], 2, 2, 4, 3, True, (-1, -1), False),
    ([0, 6], [0, 6], 4, 2, 4, 4, True, (-1, -1), False),
    ([0, 7], [0, 7], 2, 2, 3, 3, True, (2, 0), False),
    ([0, 3, 3, 8], [0, 3, 3, 8], 2, 1, 4, 2, True, (-1, -1), False),
    ([0, 4], [0, 7], 2, 2, 3, 3, True, (-1, -1), True),
    ([0, 5], [0, 5], 2, 2, 3, 3, False, (1, 1), False),
]


@pytest.mark.parametrize("case", FD_CASES)
def test_backward_finite_differences(case):
    cu_q, cu_k, hq, hkv, dqk, dv, causal, window, br = case
    tq, tk = cu_q[-1], cu_k[-1]
    q, k, v = rand(tq, hq, dqk), rand(tk, hkv, dqk), rand(tk, hkv, dv)
    do = rand(tq, hq, dv)
    kw = dict(scale=0.7, causal=causal, window=window, bottom_right=br)
    dq, dk, dvv = oracle.bwd(q, k, v, do, cu_q, cu_k, **kw)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], do, cu_q, cu_k, **kw)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], do, cu_q, cu_k, **kw)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - g)) / max(1e-12, np.max(np.abs(g)))
        assert err < 1e-6, (name, err)


def test_causal_row0_returns_v0():
    q, k, v = rand(11, 3, 8), rand(11, 3, 8), rand(11, 3, 5)
    o, lse = oracle.fwd(q, k, v, [0, 11], [0, 11], scale=0.4, causal=True)
    np.testing.assert_array_equal(o[0], v[0])
    np.testing.assert_allclose(lse[:, 0], 0.4 * np.sum(q[0] * k[0], axis=-1), atol=1e-14)


@pytest.mark.parametrize("wl", [-1, 0, 3])
def test_q_zero_closed_form(wl):
    """Q = 0 gives uniform attention over the visible keys."""
    n, d = 12, 5
    q = np.zeros((n, 1, d))
    k, v, do = rand(n, 1, d), rand(n, 1, 4), rand(n, 1, 4)
    kw = dict(scale=0.5, causal=True, window=(wl, 0))
    o, lse = oracle.fwd(q, k, v, [0, n], [0, n], **kw)
    dq, dk, dvv = oracle.bwd(q, k, v, do, [0, n], [0, n], **kw)
    for i in range(n):
        lo = 0 if wl < 0 else max(0, i - wl)
        cnt = i - lo + 1
        np.testing.assert_allclose(o[i, 0], v[lo:i + 1, 0].mean(axis=0), atol=1e-14)
        assert abs(lse[0, i] - math.log(cnt)) < 1e-14
    for j in range(n):
        exp_dv = np.zeros(4)
        for i in range(n):
            lo = 0 if wl < 0 else max(0, i - wl)
            if lo <= j <= i:
                exp_dv += do[i, 0] / (i - lo + 1)
        np.testing.assert_allclose(dvv[j, 0], exp_dv, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)


def test_dk_sums_to_zero():
    q, k, v, do = rand(20, 4, 6), rand(20, 2, 6), rand(20, 2, 6), rand(20, 4, 6)
    _, dk, _ = oracle.bwd(q, k, v, do, [0, 20], [0, 20], scale=0.3, causal=True)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)


def test_key_shift_invariance():
    q, k, v = rand(15, 2, 6), rand(15, 2, 6), rand(15, 2, 4)
    c = rand(6)
    o1, l1 = oracle.fwd(q, k, v, [0, 15], [0, 15], scale=0.6, causal=True)
    o2, l2 = oracle.fwd(q, k + c, v, [0, 15], [0, 15], scale=0.6, causal=True)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + 0.6 * np.einsum("thd,d->ht", q, c), atol=1e-12)


def test_gqa_equals_repeated_mha():
    q, k, v, do = rand(14, 6, 8), rand(14, 2, 8), rand(14, 2, 4), rand(14, 6, 4)
    kw = dict(scale=0.35, causal=True)
    o, lse = oracle.fwd(q, k, v, [0, 14], [0, 14], **kw)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    o2, lse2 = oracle.fwd(q, kr, vr, [0, 14], [0, 14], **kw)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)
    dq, dk, dvv = oracle.bwd(q, k, v, do, [0, 14], [0, 14], **kw)
    dq2, dk2, dv2 = oracle.bwd(q, kr, vr, do, [0, 14], [0, 14], **kw)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(14, 2, 3, 8).sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(dvv, dv2.reshape(14, 2, 3, 4).sum(axis=2), atol=1e-13)


def test_thd_equals_per_document():
    lens = [5, 0, 9, 1, 7]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    t = int(cu[-1])
    q, k, v, do = rand(t, 4, 8), rand(t, 2, 8), rand(t, 2, 8), rand(t, 4, 8)
    kw = dict(scale=0.3, causal=True, window=(3, 0))
    o, lse = oracle.fwd(q, k, v, cu, cu, **kw)
    dq, dk, dvv = oracle.bwd(q, k, v, do, cu, cu, **kw)
    for b, n in enumerate(lens):
        s = slice(cu[b], cu[b + 1])
        if n == 0:
            continue
        ob, lb = oracle.fwd(q[s], k[s], v[s], [0, n], [0, n], **kw)
        gq, gk, gv = oracle.bwd(q[s], k[s], v[s], do[s], [0, n], [0, n], **kw)
        np.testing.assert_allclose(o[s], ob, atol=1e-14)
        np.testing.assert_allclose(lse[:, s], lb, atol=1e-14)
        np.testing.assert_allclose(dq[s], gq, atol=1e-14)
        np.testing.assert_allclose(dk[s], gk, atol=1e-14)
        np.testing.assert_allclose(dvv[s], gv, atol=1e-14)


def test_window_limits():
    n = 16
    q, k, v = rand(n, 2, 4), rand(n, 2, 4), rand(n, 2, 3)
    kw = dict(scale=0.5)
    o00, lse00 = oracle.fwd(q, k, v, [0, n], [0, n], causal=False, window=(0, 0), **kw)
    np.testing.assert_array_equal(o00, v)  # each query sees only its own key
    oc, lc = oracle.fwd(q, k, v, [0, n], [0, n], causal=True, **kw)
    ow, lw = oracle.fwd(q, k, v, [0, n], [0, n], causal=True, window=(n, 0), **kw)
    np.testing.assert_array_equal(oc, ow)
    np.testing.assert_array_equal(lc, lw)
    o3, _ = oracle.fwd(q, k, v, [0, n], [0, n], causal=True, window=(3, 0), **kw)
    assert np.max(np.abs(o3 - oc)) > 1e-3  # a dropped window bound would be visible


def test_bottom_right_equals_tail_of_square():
    lq, lk = 6, 14
    q, k, v = rand(lk, 2, 8), rand(lk, 2, 8), rand(lk, 2, 8)
    full_o, full_l = oracle.fwd(q, k, v, [0, lk], [0, lk], scale=0.4, causal=True)
    o, lse = oracle.fwd(q[lk - lq:], k, v, [0, lq], [0, lk], scale=0.4, causal=True,
                        bottom_right=True)
    np.testing.assert_allclose(o, full_o[lk - lq:], atol=1e-14)
    np.testing.assert_allclose(lse, full_l[:, lk - lq:], atol=1e-14)


def test_keyless_rows_zero():
    """Bottom-right causal with Sq > Sk: the first Sq-Sk rows see no key."""
    lq, lk = 9, 4
    q, k, v, do = rand(lq, 2, 8), rand(lk, 2, 8), rand(lk, 2, 8), rand(lq, 2, 8)
    kw = dict(scale=0.4, causal=True, bottom_right=True)
    o, lse = oracle.fwd(q, k, v, [0, lq], [0, lk], **kw)
    dq, _, _ = oracle.bwd(q, k, v, do, [0, lq], [0, lk], **kw)
    assert np.all(o[: lq - lk] == 0.0)
    assert np.all(np.isneginf(lse[:, : lq - lk]))
    assert np.all(dq[: lq - lk] == 0.0)
    assert np.all(np.isfinite(lse[:, lq - lk:]))


def _dual_chunk_pieces(s, cp):
    """Ring-step pieces of the dual-chunk-swap causal partition.

    Rank r holds chunks r and 2cp-1-r; at step t it sees the key chunks of rank
    (r - t) mod cp.  Returns a list of (q_rows, k_rows, causal) in global rows."""
    c = s // (2 * cp)
    chunk = lambda i: np.arange(i * c, (i + 1) * c)  # noqa: E731
    pieces = []
    for r in range(cp):
        local_q = np.concatenate([chunk(r), chunk(2 * cp - 1 - r)])
        for t in range(cp):
            src = (r - t) % cp
            local_k = np.concatenate([chunk(src), chunk(2 * cp - 1 - src)])
            if t == 0:
                pieces.append((local_q, local_k, True))
            elif src < r:
                pieces.append((local_q, chunk(src), False))
            else:
                pieces.append((chunk(2 * cp - 1 - r), local_k, False))
    return pieces


def test_lse_merge_of_ring_partials_equals_full():
    s, hq, d = 64, 2, 8
    q, k, v = rand(s, hq, d), rand(s, hq, d), rand(s, hq, 6)
    full_o, full_l = oracle.fwd(q, k, v, [0, s], [0, s], scale=0.3, causal=True)
    # group pieces by query row set and merge per query row
    parts_o = np.zeros((0, s, hq, 6))
    parts_l = np.zeros((0, hq, s))
    for qr, kr, causal in _dual_chunk_pieces(s, 8):
        o, lse = oracle.fwd(q[qr], k[kr], v[kr], [0, len(qr)], [0, len(kr)], scale=0.3,
                            causal=causal)
        po = np.zeros((1, s, hq, 6))
        pl = np.full((1, hq, s), -np.inf)
        po[0, qr] = o
        pl[0][:, qr] = lse
        parts_o = np.concatenate([parts_o, po])
        parts_l = np.concatenate([parts_l, pl])
    o, lse = oracle.lse_merge(parts_o, parts_l)
    np.testing.assert_allclose(o, full_o, atol=1e-12)
    np.testing.assert_allclose(lse, full_l, atol=1e-12)


def test_lse_merge_of_chunk_pairs_equals_full():
    s, nc = 48, 6
    q, k, v = rand(s, 1, 4), rand(s, 1, 4), rand(s, 1, 3)
    full_o, full_l = oracle.fwd(q, k, v, [0, s], [0, s], scale=0.8, causal=True)
    c = s // nc
    for a in range(nc):
        qr = slice(a * c, (a + 1) * c)
        pos, pls = [], []
        for b in range(a + 1):
            kr = slice(b * c, (b + 1) * c)
            o, lse = oracle.fwd(q[qr], k[kr], v[kr], [0, c], [0, c], scale=0.8, causal=(a == b))
            pos.append(o)
            pls.append(lse)
        o, lse = oracle.lse_merge(np.stack(pos), np.stack(pls))
        np.testing.assert_allclose(o, full_o[qr], atol=1e-12)
        np.testing.assert_allclose(lse, full_l[:, qr], atol=1e-12)


@pytest.mark.parametrize("wl", [-1, 5])
def test_allgather_trimmed_calls_equal_full(wl):
    """All-gather CP decomposition: per query chunk, the trimmed key range with
    bottom-right causal alignment (and the same window) reproduces the full
    causal attention exactly; the per-chunk dK/dV partials sum to the full
    dK/dV (TransformerEngine PR #3527 review notes on all_gather)."""
    from bwd_tcgen05_tmem_gb300 import cp as cpmod
    s, ncp, hq, hkv = 48, 3, 2, 1
    q, k, v, do = rand(s, hq, 8), rand(s, hkv, 8), rand(s, hkv, 6), rand(s, hq, 6)
    kw = dict(scale=0.4, causal=True, window=(wl, -1))
    full_o, full_l = oracle.fwd(q, k, v, [0, s], [0, s], **kw)
    fdq, fdk, fdv = oracle.bwd(q, k, v, do, [0, s], [0, s], **kw)
    c = s // (2 * ncp)
    dk, dv = np.zeros_like(fdk), np.zeros_like(fdv)
    seen = np.zeros(s, dtype=bool)
    for pcs in cpmod.allgather_pieces(ncp, c, wl):
        for r, (q0, nq), (k0, k1) in pcs:
            # local row q0 of rank r is global chunk r (q0 = 0) or 2cp-1-r (q0 = c)
            g0 = (r if q0 == 0 else 2 * ncp - 1 - r) * c
            qr = slice(g0, g0 + nq)
            kr = slice(k0, k1)
            kwp = dict(kw, bottom_right=True)
            o, lse = oracle.fwd(q[qr], k[kr], v[kr], [0, nq], [0, k1 - k0], **kwp)
            pdq, pdk, pdv = oracle.bwd(q[qr], k[kr], v[kr], do[qr], [0, nq], [0, k1 - k0], **kwp)
            np.testing.assert_allclose(o, full_o[qr], atol=1e-12)
            np.testing.assert_allclose(lse, full_l[:, qr], atol=1e-12)
            np.testing.assert_allclose(pdq, fdq[qr], atol=1e-12)
            dk[kr] += pdk
            dv[kr] += pdv
            seen[qr] = True
    assert seen.all()  # the chunks cover every query row exactly
    np.testing.assert_allclose(dk, fdk, atol=1e-12)
    np.testing.assert_allclose(dv, fdv, atol=1e-12)


def test_lse_merge_neg_inf_parts():
    o_parts = rand(3, 4, 2, 5)
    l_parts = rand(3, 2, 4)
    l_parts[1] = -np.inf           # part 1 is empty everywhere
    l_parts[:, 0, 2] = -np.inf     # row 2 of head 0 is empty in all parts
    o, lse = oracle.lse_merge(o_parts, l_parts)
    o2, lse2 = oracle.lse_merge(o_parts[[0, 2]], l_parts[[0, 2]])
    np.testing.assert_allclose(o[:, 1], o2[:, 1], atol=1e-14)
    assert np.isneginf(lse[0, 2]) and np.all(o[2, 0] == 0.0)
    # two parts: closed form of the weights
    a, b = l_parts[0, 1, 0], l_parts[2, 1, 0]
    w = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(o[0, 1], w * o_parts[0, 0, 1] + (1 - w) * o_parts[2, 0, 1],
                               atol=1e-14)
    assert abs(lse[1, 0] - math.log(math.exp(a) + math.exp(b))) < 1e-14


def test_golden_two_key_example():
    """Hand-derived values (tests/golden/two_key_example.json)."""
    with open(os.path.join(GOLDEN, "two_key_example.json")) as f:
        g = json.load(f)
    q = np.array(g["q"])[:, None, :]
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    do = np.array(g["dout"])[:, None, :]
    n = q.shape[0]
    o, lse = oracle.fwd(q, k, v, [0, n], [0, n], scale=g["scale"], causal=True)
    dq, dk, dvv = oracle.bwd(q, k, v, do, [0, n], [0, n], scale=g["scale"], causal=True)
    np.testing.assert_allclose(o[:, 0], g["o"], atol=1e-14)
    np.testing.assert_allclose(lse[0], g["lse"], atol=1e-14)
    np.testing.assert_allclose(dq[:, 0], g["dq"], atol=1e-14)
    np.testing.assert_allclose(dk[:, 0], g["dk"], atol=1e-14)
    np.testing.assert_allclose(dvv[:, 0], g["dv"], atol=1e-14)


# ---------------------------------------------------------------- accuracy floor
def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).float().numpy()


def test_naive_without_rounding_matches_oracle():
    q, k, v, do = (rand(40, 2, 16) for _ in range(4))
    kw = dict(scale=0.25, causal=True)
    o, lse, dq, dk, dvv = oracle.naive(q, k, v, [0, 40], [0, 40], dtype="fp32", dout=do, **kw)
    eo, el = oracle.fwd(q, k, v, [0, 40], [0, 40], **kw)
    gq, gk, gv = oracle.bwd(q, k, v, do, [0, 40], [0, 40], **kw)
    for a, b in ((o, eo), (lse, el), (dq, gq), (dk, gk), (dvv, gv)):
        np.testing.assert_allclose(a, b, atol=5e-5)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_two_x_criterion_and_mutation(dtype):
    """Rounded exact output passes the 2x gate; a 1 % scale error does not."""
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    cast = lambda x: torch.tensor(x, dtype=torch.float32).to(tdt).float().numpy()  # noqa
    s, h, d = 256, 2, 64
    q, k, v, do = (cast(rand(s, h, d)) for _ in range(4))
    scale = 1.0 / 8
    kw = dict(causal=True)
    eo, _ = oracle.fwd(q, k, v, [0, s], [0, s], scale=scale, **kw)
    gq, gk, gv = oracle.bwd(q, k, v, do, [0, s], [0, s], scale=scale, **kw)
    no, _, nq, nk, nv = oracle.naive(q, k, v, [0, s], [0, s], scale=scale, dtype=dtype,
                                     dout=do, **kw)
    floors = [np.max(np.abs(a - b)) for a, b in ((no, eo), (nq, gq), (nk, gk), (nv, gv))]
    assert all(1e-5 < f < 0.1 for f in floors), floors
    good = [cast(x) for x in (eo, gq, gk, gv)]
    exact = (eo, gq, gk, gv)
    for x, e, f in zip(good, exact, floors):
        assert np.max(np.abs(x - e)) <= 2 * f
    mo, _ = oracle.fwd(q, k, v, [0, s], [0, s], scale=scale * 1.01, **kw)
    mq, mk, mv = oracle.bwd(q, k, v, do, [0, s], [0, s], scale=scale * 1.01, **kw)
    rejected = [np.max(np.abs(cast(x) - e)) > 2 * f
                for x, e, f in zip((mo, mq, mk, mv), exact, floors)]
    assert any(rejected), rejected
    if dtype == "fp16":
        assert all(rejected), rejected  # fp16's finer mantissa exposes it everywhere


def test_a2a_head_shards_equal_full():
    """All-to-all CP: rank r attends over the whole sequence with query heads
    [r*hq/cp, ...) and kv heads [r*hkv/cp, ...); with GQA the local group map
    h_local -> h_local // (hq/hkv) is the global one restricted to the rank."""
    s, hq, hkv, ncp = 20, 8, 4, 2
    q, k, v, do = rand(s, hq, 6), rand(s, hkv, 6), rand(s, hkv, 5), rand(s, hq, 5)
    kw = dict(scale=0.5, causal=True, window=(7, -1))
    fo, fl = oracle.fwd(q, k, v, [0, s], [0, s], **kw)
    fdq, fdk, fdv = oracle.bwd(q, k, v, do, [0, s], [0, s], **kw)
    a, b = hq // ncp, hkv // ncp
    for r in range(ncp):
        hs, gs = slice(r * a, (r + 1) * a), slice(r * b, (r + 1) * b)
        o, lse = oracle.fwd(q[:, hs], k[:, gs], v[:, gs], [0, s], [0, s], **kw)
        dq, dk, dv = oracle.bwd(q[:, hs], k[:, gs], v[:, gs], do[:, hs], [0, s], [0, s], **kw)
        np.testing.assert_array_equal(o, fo[:, hs])
        np.testing.assert_array_equal(lse, fl[hs])
        np.testing.assert_allclose(dq, fdq[:, hs], atol=1e-14)
        np.testing.assert_allclose(dk, fdk[:, gs], atol=1e-14)
        np.testing.assert_allclose(dv, fdv[:, gs], atol=1e-14)


@pytest.mark.parametrize("ncp", [1, 2, 3, 4, 8])
def test_ring_pieces_cover_every_causal_pair_once(ncp):
    """The p2p ring schedule of the CP emulation: over all ranks and steps, every
    causally visible (query, key) pair of the global sequence is computed by
    exactly one piece, with the piece's causal flag set exactly when it holds
    the diagonal (the rank's own chunk pair at step 0)."""
    from bwd_tcgen05_tmem_gb300 import cp as cpmod
    c = 5
    s = 2 * ncp * c
    local = lambda r: np.concatenate([np.arange(r * c, (r + 1) * c),  # noqa: E731
                                      np.arange((2 * ncp - 1 - r) * c, (2 * ncp - r) * c)])
    count = np.zeros((s, s), dtype=int)
    for pcs in cpmod.ring_pieces(ncp, c):
        for pc in pcs:
            qg = local(pc.rank)[pc.q_rows[0]:pc.q_rows[0] + pc.q_rows[1]]
            kg = local(pc.src)[pc.k_rows[0]:pc.k_rows[0] + pc.k_rows[1]]
            for a, i in enumerate(qg):
                for b_, j in enumerate(kg):
                    # visibility inside the piece: causal pieces are top-left over the
                    # rank's local concatenation, full pieces see every key
                    if not pc.causal or b_ <= a:
                        count[i, j] += 1
            if pc.causal:
                assert pc.rank == pc.src
            else:  # a full piece lies entirely below the diagonal
                assert qg.min() > kg.max()
    expect = np.tril(np.ones((s, s), dtype=int))
    np.testing.assert_array_equal(count, expect)


# ---------------------------------------------------------------- subsets
# The head / group / key-row selections the full-size GPU tests use to keep the
# oracle's cost down: each must give torch's float64 autograd values on what it
# selects and leave the rest untouched.


def test_head_and_group_selection_match_torch():
    s, hq, hkv, d = 23, 6, 3, 8
    q, k, v, do = rand(s, hq, d), rand(s, hkv, d), rand(s, hkv, d), rand(s, hq, d)
    kw = dict(scale=0.4, causal=True, window=(9, -1))
    o_t, lse_t, dq_t, dk_t, dv_t = torch_ref(q, k, v, dout=do, **kw)
    o, lse = oracle.fwd(q, k, v, [0, s], [0, s], heads=[1, 4], **kw)
    np.testing.assert_allclose(o[:, [1, 4]], o_t[:, [1, 4]], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[[1, 4]], lse_t[[1, 4]], rtol=0, atol=1e-12)
    assert np.all(o[:, [0, 2, 3, 5]] == 0) and np.all(np.isnan(lse[[0, 2, 3, 5]]))
    dq, dk, dvv = oracle.bwd(q, k, v, do, [0, s], [0, s], groups=[2], **kw)
    np.testing.assert_allclose(dq[:, 4:6], dq_t[:, 4:6], rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk[:, 2], dk_t[:, 2], rtol=0, atol=1e-11)
    np.testing.assert_allclose(dvv[:, 2], dv_t[:, 2], rtol=0, atol=1e-11)
    assert np.all(dq[:, :4] == 0) and np.all(dk[:, :2] == 0) and np.all(dvv[:, :2] == 0)


KV_CASES = [
    # (L, hq, hkv, causal, window, bottom_right (Lq != Lk))
    (600, 2, 1, True, (-1, -1), None),
    (600, 4, 2, True, (90, 0), None),
    (520, 2, 2, False, (70, 40), None),
    (300, 2, 1, True, (-1, -1), 450),
]


@pytest.mark.parametrize("case", KV_CASES)
def test_bwd_kv_matches_torch_autograd(case):
    """Selected key rows (first, middle and last blocks; several row blocks of
    work per head) equal torch's float64 gradients; other rows stay 0."""
    lq, hq, hkv, causal, window, lk = case
    lk = lk or lq
    d, dv = 12, 8
    q, k, v, do = rand(lq, hq, d), rand(lk, hkv, d), rand(lk, hkv, dv), rand(lq, hq, dv)
    br = lk != lq
    kw = dict(scale=0.3, causal=causal, window=window, bottom_right=br)
    _, _, _, dk_t, dv_t = torch_ref(q, k, v, dout=do, **kw)
    rows = list(range(0, 5)) + list(range(lk // 2, lk // 2 + 7)) + [lk - 1]
    dk, dvv = oracle.bwd_kv(q, k, v, do, [0, lq], [0, lk], key_rows=rows, **kw)
    np.testing.assert_allclose(dk[rows], dk_t[rows], rtol=0, atol=1e-11)
    np.testing.assert_allclose(dvv[rows], dv_t[rows], rtol=0, atol=1e-11)
    other = np.setdiff1d(np.arange(lk), rows)
    assert np.all(dk[other] == 0) and np.all(dvv[other] == 0)
    # a group selection computes only that kv head
    dk1, _ = oracle.bwd_kv(q, k, v, do, [0, lq], [0, lk], key_rows=rows, groups=[hkv - 1], **kw)
    np.testing.assert_allclose(dk1[rows, hkv - 1], dk_t[rows, hkv - 1], rtol=0, atol=1e-11)
    if hkv > 1:
        assert np.all(dk1[:, 0] == 0)


def test_bwd_kv_thd_equals_per_document_torch():
    lens = [0, 300, 1, 280]
    cu = np.cumsum([0] + lens)
    t, hq, hkv, d = cu[-1], 2, 1, 8
    q, k, v, do = rand(t, hq, d), rand(t, hkv, d), rand(t, hkv, d), rand(t, hq, d)
    rows = [1, 2, 299, 300, 301, 302, 580]
    dk, dvv = oracle.bwd_kv(q, k, v, do, cu, cu, key_rows=rows, scale=0.35, causal=True)
    for b in range(len(lens)):
        a, e = cu[b], cu[b + 1]
        if e == a:
            continue
        _, _, _, dk_t, dv_t = torch_ref(q[a:e], k[a:e], v[a:e], dout=do[a:e], scale=0.35,
                                        causal=True)
        sel = [r - a for r in rows if a <= r < e]
        np.testing.assert_allclose(dk[a:e][sel], dk_t[sel], rtol=0, atol=1e-11)
        np.testing.assert_allclose(dvv[a:e][sel], dv_t[sel], rtol=0, atol=1e-11)


def test_naive_kv_without_rounding_matches_exact_and_floor_works():
    """No rounding (FP32 type): naive_kv equals the exact subset to FP32
    accuracy.  With BF16 its floor accepts the rounded exact dK/dV of the
    selected rows and rejects a 1 % softmax-scale error (TransformerEngine
    PR #3527's mutation test, on a key subset)."""
    s, hq, hkv, d = 700, 2, 1, 16
    q, k, v, do = (_bf16(rand(s, h, d)) for h in (hq, hkv, hkv, hq))
    rows = list(range(0, 128)) + list(range(400, 420))
    kw = dict(scale=0.25, causal=True, key_rows=rows)
    ek, ev = oracle.bwd_kv(q, k, v, do, [0, s], [0, s], **kw)
    fk, fv = oracle.naive_kv(q, k, v, do, [0, s], [0, s], dtype="fp32", **kw)
    np.testing.assert_allclose(fk[rows], ek[rows], atol=5e-5)
    np.testing.assert_allclose(fv[rows], ev[rows], atol=5e-5)
    nk, nv = oracle.naive_kv(q, k, v, do, [0, s], [0, s], dtype="bf16", **kw)
    floors = [np.max(np.abs(nk[rows] - ek[rows])), np.max(np.abs(nv[rows] - ev[rows]))]
    assert all(1e-5 < f < 0.1 for f in floors), floors
    for x, e, f in ((ek, ek, floors[0]), (ev, ev, floors[1])):
        assert np.max(np.abs(_bf16(x[rows]) - e[rows])) <= 2 * f
    mk, mv = oracle.bwd_kv(q, k, v, do, [0, s], [0, s], scale=0.25 * 1.01, causal=True,
                           key_rows=rows)
    rejected = [np.max(np.abs(_bf16(m[rows]) - e[rows])) > 2 * f
                for m, e, f in ((mk, ek, floors[0]), (mv, ev, floors[1]))]
    assert any(rejected), rejected
